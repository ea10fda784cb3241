#!/usr/bin/env python
"""Benchmark of the NVFP4 dense-MLP hot path on one GB300 (or N replicas).

Workload: the decode dense MLP, W4A4 NVFP4, hidden 5120, intermediate 17408
(gate_up 34816 x 5120, down 5120 x 17408).  One step runs the MLP forward
once for each decode batch M in {1, 2, 4, 8, 16} (31 tokens per step):
    nvfp4_quantize(x) -> nvfp4_gemm(gate_up) -> silu_mul_nvfp4_quantize
    -> nvfp4_gemm(down)
Weights are synthetic N(0, 0.02), quantized to NVFP4 on the device by the
library before timing; x ~ N(0, 1) bf16.  Each step's launches are captured
in a CUDA graph; four weight copies (602 MB, > 4x the 126 MB L2) rotate so the
weight stream comes from HBM every step.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on
the host cores instead (the slow baseline arm).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

H, I = 5120, 17408
MS = (1, 2, 4, 8, 16)
TOKENS_PER_STEP = sum(MS)
NCOPY = 4
METRIC = "NVFP4 MLP tokens/s (decode H5120 I17408, M in 1,2,4,8,16)"
WORKLOAD = "decode dense MLP W4A4 NVFP4, hidden 5120, intermediate 17408, M sweep 1/2/4/8/16"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------- oracle leg
def oracle_sample(ms, seconds_cap=None):
    """Time the CPU oracle's unfused decode MLP at the given M values (same
    shapes and recipe; weights quantized beforehand, not timed).  Returns
    (tokens, seconds, threads)."""
    import numpy as np
    import oracle
    import synth

    wgu, wdn = synth.weight(1, "gate_up"), synth.weight(1, "down")
    gs_gu = oracle.global_scale(np.abs(wgu).max())
    gs_dn = oracle.global_scale(np.abs(wdn).max())
    gu = oracle.quantize_nvfp4(wgu, gs_gu)
    dn = oracle.quantize_nvfp4(wdn, gs_dn)
    del wgu, wdn
    tokens, secs = 0, 0.0
    for m in ms:
        _, x = synth.activations(1, m)
        gs_x = oracle.global_scale(np.abs(x).max())
        a_gu = np.float32(1.0) / (gs_x * gs_gu)
        gs_h = np.float32(448.0 * 6.0 / 8.0)
        a_dn = np.float32(1.0) / (gs_h * gs_dn)
        t0 = time.perf_counter()
        oracle.mlp_w4a4_unfused(x, gs_x, gu, a_gu, gs_h, dn, a_dn)
        secs += time.perf_counter() - t0
        tokens += m
        if seconds_cap and secs > seconds_cap:
            break
    threads = os.cpu_count()
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        threads = max([i.get("num_threads", 1) for i in info] or [threads])
    except Exception:
        pass
    return tokens, secs, threads


def run_reference(args, world, rank):
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample((16,))
    tokens, secs = 0, 0.0
    threads = os.cpu_count()
    for _ in range(args.steps):
        t, s, threads = oracle_sample((16,))
        tokens += t
        secs += s
    value = tokens / secs
    sample = "CPU oracle (NumPy float64), one decode MLP forward at M=16 per step, H5120 I17408"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "step": "M=16 forward (bounded sample)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU leg
class Clocks:
    """nvidia-smi sampler over the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        self.proc.wait()
        self.out.close()
        rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.strip()]
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            if len(r) < 9:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(rows)}


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import nvfp4_quantized_dense_gb300 as nv

    nv.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)

    def scalar(v):
        return torch.tensor([np.float32(v)], dtype=torch.float32, device=dev)

    def gscale(t):
        return np.float32(np.float32(448.0 * 6.0) / np.float32(t.abs().max().float().item()))

    def make_weight(rows, cols):
        w = (torch.randn(rows, cols, generator=gen, device=dev) * 0.02).to(torch.bfloat16)
        gs = gscale(w)
        q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        s_lin = torch.empty((rows * cols // 16,), dtype=torch.uint8, device=dev)
        nv.nvfp4_quantize(w, rows, cols, scalar(gs), q, s_lin, nv.SF_LINEAR)
        s = torch.empty((nv.nvfp4_sf_bytes(rows, cols),), dtype=torch.uint8, device=dev)
        nv.nvfp4_prepare_weights(q, s_lin, rows, cols, q, s)
        del w, s_lin
        return q, s, gs

    wgu0 = make_weight(2 * I, H)
    wdn0 = make_weight(H, I)
    copies = [(wgu0, wdn0)]
    for _ in range(NCOPY - 1):
        copies.append(((wgu0[0].clone(), wgu0[1].clone(), wgu0[2]), (wdn0[0].clone(), wdn0[1].clone(), wdn0[2])))
    weight_bytes = sum(t.numel() for t in (wgu0[0], wgu0[1], wdn0[0], wdn0[1]))

    mmax = max(MS)
    x = torch.randn(mmax, H, generator=gen, device=dev).to(torch.bfloat16)
    gs_x = gscale(x)
    # calibrate the static down_proj input scale once from the gate_up output
    gu_tmp = torch.empty((mmax, 2 * I), dtype=torch.bfloat16, device=dev)
    xq = torch.empty((mmax, H // 2), dtype=torch.uint8, device=dev)
    xs = torch.empty((nv.nvfp4_sf_bytes(mmax, H),), dtype=torch.uint8, device=dev)
    nv.nvfp4_quantize(x, mmax, H, scalar(gs_x), xq, xs)
    a_gu = scalar(np.float32(1.0) / (gs_x * wgu0[2]))
    nv.nvfp4_gemm(xq, xs, wgu0[0], wgu0[1], a_gu, gu_tmp, mmax, 2 * I, H)
    g, u = gu_tmp.float()[:, :I], gu_tmp.float()[:, I:]
    gs_h = gscale(g * torch.sigmoid(g) * u)
    a_dn = scalar(np.float32(1.0) / (gs_h * wdn0[2]))
    gs_x_d, gs_h_d = scalar(gs_x), scalar(gs_h)
    del gu_tmp

    # per-M buffers
    bufs = {}
    for m in MS:
        bufs[m] = dict(
            xq=torch.empty((m, H // 2), dtype=torch.uint8, device=dev),
            xs=torch.empty((nv.nvfp4_sf_bytes(m, H),), dtype=torch.uint8, device=dev),
            gu=torch.empty((m, 2 * I), dtype=torch.bfloat16, device=dev),
            hq=torch.empty((m, I // 2), dtype=torch.uint8, device=dev),
            hs=torch.empty((nv.nvfp4_sf_bytes(m, I),), dtype=torch.uint8, device=dev),
            out=torch.empty((m, H), dtype=torch.bfloat16, device=dev))
    x_in = {m: x[:m].contiguous() for m in MS}

    try:
        torch.cuda.Event(enable_timing=True, external=True)
        ext_ok = True
    except TypeError:
        ext_ok = False

    def forward(m, wc, ev=None):
        b = bufs[m]
        (gq, gsf, _), (dq, dsf, _) = wc
        nv.nvfp4_quantize(x_in[m], m, H, gs_x_d, b["xq"], b["xs"])
        if ev is not None:
            ev[0].record()
        nv.nvfp4_gemm(b["xq"], b["xs"], gq, gsf, a_gu, b["gu"], m, 2 * I, H)
        if ev is not None:
            ev[1].record()
        nv.silu_mul_nvfp4_quantize(b["gu"], m, I, gs_h_d, b["hq"], b["hs"])
        nv.nvfp4_gemm(b["hq"], b["hs"], dq, dsf, a_dn, b["out"], m, H, I)

    launches_per_step = 4 * len(MS)

    # capture one graph per weight copy, with timing events around gate_up
    stream = torch.cuda.Stream(device=dev)
    graphs, events = [], []
    with torch.cuda.stream(stream):
        for m in MS:                      # warm the kernels outside capture
            forward(m, copies[0])
        torch.cuda.synchronize()
        for c in range(NCOPY):
            evs = [(torch.cuda.Event(enable_timing=True, external=True),
                    torch.cuda.Event(enable_timing=True, external=True)) for _ in MS] if ext_ok else None
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                for j, m in enumerate(MS):
                    forward(m, copies[c], evs[j] if evs else None)
            graphs.append(gr)
            events.append(evs)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for i in range(args.warmup):
        with torch.cuda.stream(stream):
            graphs[i % NCOPY].replay()
    torch.cuda.synchronize()

    clocks = Clocks(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    gate_ms = []
    with torch.cuda.stream(stream):
        t_start.record()
        for i in range(args.steps):
            graphs[i % NCOPY].replay()
        t_end.record()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    step_ms = t_start.elapsed_time(t_end) / args.steps
    if ext_ok:
        for c in range(min(NCOPY, args.steps)):
            gate_ms.append([events[c][j][0].elapsed_time(events[c][j][1]) for j in range(len(MS))])

    if world > 1:
        t = torch.tensor([step_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        step_ms = float(t.item())
    value = world * TOKENS_PER_STEP / (step_ms / 1000.0)

    # dominant kernel: the gate_up GEMM (weight stream 34816 x 5120 NVFP4)
    gu_bytes = lambda m: 2 * I * H // 2 + (2 * I) * H // 16 + m * H // 2 + m * H // 16 + m * 2 * I * 2
    if gate_ms:
        per_m = [statistics.mean(col) for col in zip(*gate_ms)]
    else:
        per_m = None
    pk = peaks()
    hbm_peak = pk["hbm_gbs"] if pk else 6800.0
    roofline = None
    if per_m:
        tot_bytes = sum(gu_bytes(m) for m in MS)
        tot_ms = sum(per_m)
        achieved = tot_bytes / (tot_ms / 1000.0) / 1e9
        roofline = {"bound": "hbm", "kernel": "nvfp4_gemm gate_up (34816x5120), M=1..16",
                    "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak, "traffic": None,
                    "peak_source": "measured" if pk else "fallback",
                    "per_m_us": {str(m): 1000.0 * t for m, t in zip(MS, per_m)}}

    # end to end through the API: pinned host x in, host result out, per step
    x_host = x.cpu().pin_memory()
    outs_host = {m: torch.empty((m, H), dtype=torch.bfloat16).pin_memory() for m in MS}
    h2d = sum(m * H * 2 for m in MS)
    d2h = sum(m * H * 2 for m in MS)
    e2e_steps = max(3, min(args.steps, 20))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(2):
            for m in MS:
                x_in[m].copy_(x_host[:m], non_blocking=True)
                forward(m, copies[i % NCOPY])
                outs_host[m].copy_(bufs[m]["out"], non_blocking=True)
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        for i in range(e2e_steps):
            for m in MS:
                x_in[m].copy_(x_host[:m], non_blocking=True)
                forward(m, copies[i % NCOPY])
                outs_host[m].copy_(bufs[m]["out"], non_blocking=True)
        stream.synchronize()
        e2e_s = (time.perf_counter() - w0) / e2e_steps
    e2e_value = world * TOKENS_PER_STEP / e2e_s

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tokens, secs, threads = oracle_sample((1, 16))
        cpu = {"value": tokens / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": "CPU oracle (NumPy float64) decode MLP forward at M=1 and M=16, "
                         "H5120 I17408, weights pre-quantized"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "nvfp4 (e2m1 x ue4m3, fp32 accumulate)", "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens_per_step": TOKENS_PER_STEP,
                       "l2": f"{NCOPY} rotating weight copies, {NCOPY * weight_bytes / 1e6:.0f} MB > L2",
                       "graph": "one CUDA graph per step", "parallelism": f"replicas{world}"},
            "roofline": roofline, "cpu_baseline": cpu, "clocks": clk,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "note": "direct API calls, no graph, pinned host buffers"},
            "gpu_launches": launches_per_step * args.steps,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
