#!/usr/bin/env python
"""Benchmark of the NVFP4 dense-MLP hot path on one GB300 (or N replicas).

Workload: the decode dense MLP, W4A4 NVFP4, hidden 5120, intermediate 17408
(gate_up 34816 x 5120, down 5120 x 17408).  One step runs the MLP forward
once for each decode batch M in {1, 2, 4, 8, 16} (31 tokens per step) as
three launches each (the default `--decode-path chain`):
    nvfp4_quantize(x) -> nvfp4_gemm_swiglu_quant(gate_up; SwiGLU on the fp32
    accumulators + NVFP4 requantize in the epilogue) -> nvfp4_gemm(down)
both GEMMs on the weight-streaming swap-AB tensor-core kernel.
`--decode-path fused` runs each MLP as one nvfp4_mlp_decode launch instead
(SwiGLU on the bf16-rounded gate_up, as silu_mul_nvfp4_quantize).
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
    p.add_argument("--workload", default="decode", choices=["decode", "prefill", "w4a16"],
                   help="decode (default line) | prefill H7168/I18432 | w4a16 H5120/I17408")
    p.add_argument("--m", type=int, default=None, help="single M (decode: instead of the 1..16 sweep)")
    p.add_argument("--algo", default="auto", choices=["auto", "gemv", "tc", "tc1sm", "swapab"],
                   help="GEMM kernel family of the chain's GEMMs (auto: the library's choice by M; "
                        "tc: CTA pairs with 2-SM MMAs; tc1sm: one CTA per tile)")
    p.add_argument("--decode-path", default="chain", choices=["fused", "chain"],
                   help="decode MLP as three launches (default) or one nvfp4_mlp_decode launch")
    return p.parse_args()


def aggregate(step_ms, tokens_per_step, world, device=None):
    """Whole-job throughput of N independent replicas: every rank processed
    `tokens_per_step` tokens per step; the job's step time is the slowest
    rank's (max over ranks).  Returns (max step ms, tokens/s)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(step_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms = float(t.item())
    return step_ms, world * tokens_per_step / (step_ms / 1000.0)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------- oracle leg
# The CPU oracle's cost is linear in the intermediate size I (both GEMMs) and
# dominated by them, so a bounded sample runs the decode MLP on a slice of I:
# the first I/SLICE gate rows and as many up rows, and the matching I/SLICE
# input columns of down_proj (same H, same weight and activation recipe).
# Its tokens/s is scaled back to the whole MLP: tokens * (1/SLICE) / seconds.
SLICE = 8


class OracleSampler:
    def __init__(self):
        import numpy as np
        import oracle
        import synth
        self.np, self.oracle, self.synth = np, oracle, synth
        self.isl = I // SLICE
        wgu = synth.weight(1, "gate_up", rows=2 * self.isl)     # [gate slice; up slice]
        wdn = synth.weight(1, "down", cols=self.isl)
        self.gs_gu = oracle.global_scale(np.abs(wgu).max())
        self.gs_dn = oracle.global_scale(np.abs(wdn).max())
        self.gu = oracle.quantize_nvfp4(wgu, self.gs_gu)
        self.dn = oracle.quantize_nvfp4(wdn, self.gs_dn)

    def forward(self, m):
        """One timed oracle MLP forward (unfused chain) at M = m on the slice;
        returns (whole-MLP token equivalents, seconds)."""
        np, oracle = self.np, self.oracle
        _, x = self.synth.activations(1, m)
        gs_x = oracle.global_scale(np.abs(x).max())
        a_gu = np.float32(1.0) / (gs_x * self.gs_gu)
        gs_h = np.float32(448.0 * 6.0 / 8.0)
        a_dn = np.float32(1.0) / (gs_h * self.gs_dn)
        t0 = time.perf_counter()
        oracle.mlp_w4a4_unfused(x, gs_x, self.gu, a_gu, gs_h, self.dn, a_dn)
        return m / SLICE, time.perf_counter() - t0

    @staticmethod
    def threads():
        n = os.cpu_count()
        try:
            import threadpoolctl
            info = threadpoolctl.threadpool_info()
            n = max([i.get("num_threads", 1) for i in info] or [n])
        except Exception:
            pass
        return n


def oracle_sample(ms):
    """The CPU baseline beside a GPU run: one oracle forward per M in `ms`.
    Returns (token equivalents, seconds, threads)."""
    smp = OracleSampler()
    tokens, secs = 0.0, 0.0
    for m in ms:
        t, s = smp.forward(m)
        tokens += t
        secs += s
    return tokens, secs, smp.threads()


def run_reference(args, world, rank):
    if rank != 0:
        return
    smp = OracleSampler()
    for _ in range(args.warmup):
        smp.forward(16)
    tokens, secs = 0.0, 0.0
    for _ in range(args.steps):
        t, s = smp.forward(16)
        tokens += t
        secs += s
    value = tokens / secs
    sample = (f"CPU oracle (NumPy float64), per step one decode MLP forward at M=16 on a 1/{SLICE} slice of "
              f"the intermediate size (I {I // SLICE} of {I}, H {H}); tokens/s scaled to the whole MLP")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "step": f"M=16 forward on 1/{SLICE} of I (bounded sample)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": smp.threads(), "kind": "oracle",
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

    def make_weight(rows, cols, interleave=False):
        w = (torch.randn(rows, cols, generator=gen, device=dev) * 0.02).to(torch.bfloat16)
        gs = gscale(w)
        q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        s_lin = torch.empty((rows * cols // 16,), dtype=torch.uint8, device=dev)
        nv.nvfp4_quantize(w, rows, cols, scalar(gs), q, s_lin, nv.SF_LINEAR)
        s = torch.empty((nv.nvfp4_sf_bytes(rows, cols),), dtype=torch.uint8, device=dev)
        if interleave:
            qi = torch.empty_like(q)
            nv.nvfp4_prepare_gate_up_interleaved(q, s_lin, rows, cols, qi, s)
            q = qi
        else:
            nv.nvfp4_prepare_weights(q, s_lin, rows, cols, q, s)
        del w, s_lin
        return q, s, gs

    pk = peaks()
    hbm_peak = pk["hbm_gbs"] if pk else 6800.0
    bf16_peak = pk["bf16_tflops"] if pk else 1900.0
    fp4_peak = bf16_peak * 6.0        # dense FP4 : dense BF16 = 13.5 : 2.25 (nominal)

    wl = args.workload
    if wl == "decode":
        hid, inter, ms, ncopy = H, I, ((args.m,) if args.m else MS), NCOPY
        metric, workload = METRIC, WORKLOAD
        if args.m:
            metric = f"NVFP4 MLP tokens/s (decode H5120 I17408, M={args.m})"
            workload = f"decode dense MLP W4A4 NVFP4, hidden 5120, intermediate 17408, M={args.m}"
    elif wl == "prefill":
        hid, inter = 7168, 18432
        ms = (args.m or 8192,)
        ncopy = 2
        metric = f"NVFP4 MLP tokens/s (prefill H7168 I18432, M={ms[0]})"
        workload = f"prefill dense MLP W4A4 NVFP4 (fused gate_up+SwiGLU+requant), hidden 7168, intermediate 18432, M={ms[0]}"
    else:
        hid, inter = H, I
        ms = (args.m,) if args.m else (1, 16, 128, 1024)
        ncopy = NCOPY
        metric = f"W4A16 MLP tokens/s (H5120 I17408, M in {','.join(map(str, ms))})"
        workload = f"W4A16 dense MLP (bf16 x NVFP4), hidden 5120, intermediate 17408, M in {ms}"
    tokens_per_step = sum(ms)
    mmax = max(ms)
    fused_decode = wl == "decode" and args.decode_path == "fused"
    algo = {"auto": nv.ALGO_AUTO, "gemv": nv.ALGO_GEMV, "tc": nv.ALGO_TC, "tc1sm": nv.ALGO_TC_1SM,
            "swapab": nv.ALGO_TC_SWAPAB}[args.algo]
    if fused_decode and algo != nv.ALGO_AUTO:
        raise SystemExit("--algo applies to the chain of separate GEMM launches, not --decode-path fused")
    interleaved = wl in ("prefill", "decode")

    w_gu0 = make_weight(2 * inter, hid, interleave=interleaved)
    w_dn0 = make_weight(hid, inter)
    copies = [(w_gu0, w_dn0)]
    for _ in range(ncopy - 1):
        copies.append(((w_gu0[0].clone(), w_gu0[1].clone(), w_gu0[2]),
                       (w_dn0[0].clone(), w_dn0[1].clone(), w_dn0[2])))
    weight_bytes = sum(t.numel() for t in (w_gu0[0], w_gu0[1], w_dn0[0], w_dn0[1]))

    x = torch.randn(mmax, hid, generator=gen, device=dev).to(torch.bfloat16)
    gs_x = gscale(x)
    # calibrate the static down_proj input scale once from one gate_up pass
    mc = min(mmax, 1024)
    gu_tmp = torch.empty((mc, 2 * inter), dtype=torch.bfloat16, device=dev)
    if wl == "w4a16":
        nv.bf16_fp4_gemm(x[:mc].contiguous(), w_gu0[0], w_gu0[1], scalar(np.float32(1.0) / w_gu0[2]),
                         gu_tmp, mc, 2 * inter, hid)
        gs_h, a_gu = None, scalar(np.float32(1.0) / w_gu0[2])
        a_dn = scalar(np.float32(1.0) / w_dn0[2])
    else:
        xq = torch.empty((mc, hid // 2), dtype=torch.uint8, device=dev)
        xs = torch.empty((nv.nvfp4_sf_bytes(mc, hid),), dtype=torch.uint8, device=dev)
        nv.nvfp4_quantize(x[:mc].contiguous(), mc, hid, scalar(gs_x), xq, xs)
        a_gu = scalar(np.float32(1.0) / (gs_x * w_gu0[2]))
        nv.nvfp4_gemm(xq, xs, w_gu0[0], w_gu0[1], a_gu, gu_tmp, mc, 2 * inter, hid)
        gf = gu_tmp.float()
        if interleaved:       # interleaved rows: blocks of 128 = [64 up ; 64 gate]
            gf = gf.view(mc, 2 * inter // 128, 2, 64)
            u, g = gf[:, :, 0, :].reshape(mc, inter), gf[:, :, 1, :].reshape(mc, inter)
        else:
            g, u = gf[:, :inter], gf[:, inter:]
        gs_h = gscale(g * torch.sigmoid(g) * u)
        a_dn = scalar(np.float32(1.0) / (gs_h * w_dn0[2]))
    gs_x_d = scalar(gs_x)
    gs_h_d = scalar(gs_h) if gs_h is not None else None
    del gu_tmp

    # every M's output is a row range of one buffer (read back in one copy)
    out_all = torch.empty((sum(ms), hid), dtype=torch.bfloat16, device=dev)
    out_rows = {}
    r0 = 0
    for m in ms:
        out_rows[m] = out_all[r0:r0 + m]
        r0 += m
    bufs = {}
    for m in ms:
        bufs[m] = dict(
            xq=torch.empty((m, hid // 2), dtype=torch.uint8, device=dev),
            xs=torch.empty((nv.nvfp4_sf_bytes(m, hid),), dtype=torch.uint8, device=dev),
            gu=torch.empty((m, 2 * inter), dtype=torch.bfloat16, device=dev),
            h16=torch.empty((m, inter), dtype=torch.bfloat16, device=dev),
            hq=torch.empty((m, inter // 2), dtype=torch.uint8, device=dev),
            hs=torch.empty((nv.nvfp4_sf_bytes(m, inter),), dtype=torch.uint8, device=dev),
            out=out_rows[m])
    # every M's input is the first M rows of one x buffer (written in one copy)
    x_in = {m: x[:m] for m in ms}
    # one zero-filled scratch buffer (split-K partials + arrival counters),
    # sized for the largest GEMM of the chain and shared by its sequential calls
    ws_bytes = max([nv.nvfp4_workspace_bytes(m, 2 * inter, hid, algo) for m in ms] +
                   [nv.nvfp4_workspace_bytes(m, hid, inter, algo) for m in ms] + [0])
    if fused_decode:
        ws_bytes = max(nv.nvfp4_mlp_decode_workspace_bytes(m, hid, inter) for m in ms)
    if wl == "w4a16":
        ws_bytes = max([nv.bf16_fp4_gemm_workspace_bytes(m, 2 * inter, hid, algo) for m in ms] +
                       [nv.bf16_fp4_gemm_workspace_bytes(m, hid, inter, algo) for m in ms] + [0])
    ws = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

    # the stream handle as an int: the bindings then skip looking up torch's
    # current stream (~3 us of host time per call)
    SH = [None]

    def dominant(m, wc):
        """The step's dominant launch: the gate_up GEMM (the whole MLP when fused)."""
        b = bufs[m]
        (gq, gsf, _), (dq, dsf, _) = wc
        if wl == "w4a16":
            nv.bf16_fp4_gemm_ex(x_in[m], gq, gsf, a_gu, b["gu"], m, 2 * inter, hid, ws, ws_bytes, algo,
                                stream=SH[0])
        elif fused_decode:
            nv.nvfp4_mlp_decode(x_in[m], gs_x_d, gq, gsf, a_gu, gs_h_d, dq, dsf, a_dn, b["xq"], b["xs"],
                                b["hq"], b["hs"], b["out"], m, hid, inter, True, ws, ws_bytes, stream=SH[0])
        else:
            nv.nvfp4_gemm_swiglu_quant_ex(b["xq"], b["xs"], gq, gsf, a_gu, gs_h_d, b["hq"], b["hs"], m,
                                          2 * inter, hid, ws, ws_bytes, algo, stream=SH[0])

    def forward(m, wc, ev=None):
        """One MLP forward; ev = (start, end) events around the dominant kernel."""
        b = bufs[m]
        (gq, gsf, _), (dq, dsf, _) = wc
        if wl != "w4a16" and not fused_decode:
            nv.nvfp4_quantize(x_in[m], m, hid, gs_x_d, b["xq"], b["xs"], stream=SH[0])
        if ev is not None:
            ev[0].record()
        dominant(m, wc)
        if ev is not None:
            ev[1].record()
        if wl == "w4a16":
            nv.silu_mul_bf16(b["gu"], m, inter, b["h16"], stream=SH[0])
            nv.bf16_fp4_gemm_ex(b["h16"], dq, dsf, a_dn, b["out"], m, hid, inter, ws, ws_bytes, algo,
                                stream=SH[0])
        elif not fused_decode:
            nv.nvfp4_gemm_ex(b["hq"], b["hs"], dq, dsf, a_dn, b["out"], m, hid, inter, ws, ws_bytes, algo,
                             stream=SH[0])

    launches_per_step = sum((1 if fused_decode else 3) for _ in ms)

    try:
        torch.cuda.Event(enable_timing=True, external=True)
        ext_ok = True
    except TypeError:
        ext_ok = False

    stream = torch.cuda.Stream(device=dev)
    SH[0] = stream.cuda_stream
    # Two graph sets per weight copy: plain step graphs for the headline pass
    # (an event node between kernels would end their programmatic-launch
    # overlap) and the same steps with timing events around the dominant
    # kernel for the roofline pass that follows.
    graphs, probe_graphs, events = [], [], []
    with torch.cuda.stream(stream):
        for m in ms:                      # warm the kernels outside capture
            forward(m, copies[0])
        torch.cuda.synchronize()
        for c in range(ncopy):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                for m in ms:
                    forward(m, copies[c])
            graphs.append(gr)
            if ext_ok:
                evs = [(torch.cuda.Event(enable_timing=True, external=True),
                        torch.cuda.Event(enable_timing=True, external=True)) for _ in ms]
                pg = torch.cuda.CUDAGraph()
                with torch.cuda.graph(pg, stream=stream):
                    for j, m in enumerate(ms):
                        forward(m, copies[c], evs[j])
                probe_graphs.append(pg)
                events.append(evs)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for i in range(args.warmup):
        with torch.cuda.stream(stream):
            graphs[i % ncopy].replay()
    torch.cuda.synchronize()

    clocks = Clocks(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record()
        for i in range(args.steps):
            graphs[i % ncopy].replay()
        t_end.record()
    torch.cuda.synchronize()
    barrier()
    step_ms = t_start.elapsed_time(t_end) / args.steps
    # roofline pass: the same number of steps with the instrumented graphs
    dom_ms = None
    if ext_ok:
        sums = [0.0] * len(ms)
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                probe_graphs[i % ncopy].replay()
                # each graph's event nodes keep only their latest replay: read
                # them once every copy has been replayed (and at the end)
                if i % ncopy == ncopy - 1 or i == args.steps - 1:
                    stream.synchronize()
                    for c in range(i % ncopy + 1):
                        for j in range(len(ms)):
                            sums[j] += events[c][j][0].elapsed_time(events[c][j][1])
        torch.cuda.synchronize()
        dom_ms = [v / args.steps for v in sums]
    # the dominant kernel alone, REPS launches back to back in one graph
    # (weight copies rotating), events around the replays: its per-launch time
    # with the programmatic-launch overlap it also gets inside the step graph
    # (the event nodes of the pass above end that overlap)
    b2b_ms = []
    REPS = 8
    with torch.cuda.stream(stream):
        for m in ms:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                for r in range(REPS):
                    dominant(m, copies[r % ncopy])
            gr.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(3):
                gr.replay()
            e1.record(stream)
            stream.synchronize()
            b2b_ms.append(e0.elapsed_time(e1) / (3 * REPS))
            del gr
    clk = clocks.stop()

    step_ms, value = aggregate(step_ms, tokens_per_step, world, device=dev)

    roofline = None
    if b2b_ms:
        timing_note = (f"dominant-kernel time: {REPS} launches back to back in one CUDA graph per M, CUDA "
                       "events on the launching stream around 3 replays; isolated_us: events around each "
                       f"launch inside the step graphs ({args.steps}-step pass, no launch overlap)")
        per_m_us = {str(m): 1000.0 * t for m, t in zip(ms, b2b_ms)}
        tot_s = sum(b2b_ms) / 1000.0
        if fused_decode:
            # weights (codes + scales) of both GEMMs, x in, output out
            nbytes = sum(3 * inter * hid * 9 // 16 + 2 * m * hid * 2 for m in ms)
            achieved = nbytes / tot_s / 1e9
            roofline = {"bound": "hbm", "kernel": "nvfp4_mlp_decode (whole decode MLP, one launch, M=1..16)",
                        "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                        "traffic": None, "algorithmic_bytes_per_step": nbytes}
        elif wl == "decode":
            # gate_up weights (codes + scales), quantized x in, NVFP4 h out
            nbytes = sum(2 * inter * hid * 9 // 16 + m * hid * 9 // 16 + m * inter * 9 // 16 for m in ms)
            achieved = nbytes / tot_s / 1e9
            family = {"auto": "swap-AB tcgen05", "swapab": "swap-AB tcgen05", "gemv": "CUDA-core GEMV",
                      "tc": "128-token-tile tcgen05, CTA pairs", "tc1sm": "128-token-tile tcgen05"}[args.algo]
            if args.algo == "auto" and mmax > 64:
                family = "128-token-tile tcgen05"
            # traffic: DRAM bytes read + written by one launch of the swap-AB
            # NT = 16 instance (every M <= 16) in an ncu capture of this bench
            # command (summary in profiles/swapab_swiglu_gate_up_m16_h5120.md);
            # to be set to None whenever the kernel changes before it is
            # captured again
            measured = args.algo in ("auto", "swapab") and mmax <= 16
            roofline = {"bound": "hbm",
                        "kernel": f"nvfp4_gemm_swiglu_quant gate_up 34816x5120 ({family}, "
                                  f"M={','.join(map(str, ms))})",
                        "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                        "traffic": 100.42e6 + 2.94e6 if measured else None, "traffic_unit": "bytes per launch",
                        "algorithmic_bytes_per_launch": nbytes / len(ms), "algorithmic_bytes_per_step": nbytes}
        elif wl == "prefill":
            flops = sum(4.0 * m * hid * inter for m in ms)
            achieved = flops / tot_s / 1e12
            roofline = {"bound": "tensor", "kernel": "nvfp4_gemm_swiglu_quant gate_up 36864x7168 (tcgen05)",
                        "achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s", "frac": achieved / fp4_peak,
                        "traffic": None, "peak_note": "measured bf16 burst x 6 (nominal fp4:bf16)"}
        else:
            nbytes = sum(2 * inter * hid * 9 // 16 + m * hid * 2 + m * 2 * inter * 2 for m in ms)
            achieved = nbytes / tot_s / 1e9
            roofline = {"bound": "hbm", "kernel": "bf16_fp4_gemm gate_up 34816x5120",
                        "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                        "traffic": None}
        roofline["per_m_us"] = per_m_us
        if dom_ms:
            roofline["isolated_us"] = {str(m): 1000.0 * t for m, t in zip(ms, dom_ms)}
        roofline["peak_source"] = "measured" if pk else "fallback"
        roofline["timing"] = timing_note

    # end to end through the API: pinned host x in, host result out, per step
    x_host = x.cpu().pin_memory()
    out_host = torch.empty((sum(ms), hid), dtype=torch.bfloat16).pin_memory()
    h2d = x.numel() * 2
    d2h = out_all.numel() * 2
    e2e_steps = max(3, min(args.steps, 20))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        def e2e_step(i):
            x.copy_(x_host, non_blocking=True)
            for m in ms:
                forward(m, copies[i % ncopy])
            out_host.copy_(out_all, non_blocking=True)
        for i in range(2):
            e2e_step(i)
        stream.synchronize()
        w0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_step(i)
        stream.synchronize()
        e2e_s = (time.perf_counter() - w0) / e2e_steps
    e2e_value = world * tokens_per_step / e2e_s

    cpu = None
    if rank == 0 and wl == "decode" and not args.no_cpu_baseline:
        tokens, secs, threads = oracle_sample((1, 16))
        cpu = {"value": tokens / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"CPU oracle (NumPy float64) decode MLP forward at M=1 and M=16 on a 1/{SLICE} "
                         f"slice of I (I {I // SLICE} of {I}, H {H}), weights pre-quantized; tokens/s "
                         "scaled to the whole MLP"}

    if rank == 0:
        line = {
            "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16 x nvfp4 (fp32 accumulate)" if wl == "w4a16" else "nvfp4 (e2m1 x ue4m3, fp32 accumulate)",
            "data": "synthetic",
            "config": {"workload": workload, "tokens_per_step": tokens_per_step,
                       "l2": f"{ncopy} rotating weight copies, {ncopy * weight_bytes / 1e6:.0f} MB > L2",
                       "graph": "one CUDA graph per step", "parallelism": f"replicas{world}",
                       **({"decode_path": args.decode_path} if wl == "decode" else {}),
                       **({"algo": args.algo} if args.algo != "auto" else {})},
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
