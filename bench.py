#!/usr/bin/env python
"""Benchmark of the NVFP4 dense-MLP hot path on one GB300 (or N replicas).

One step runs the MLP forward once for every batch size of the four
synthetic workloads, which together span M = 1..8192:
  decode   W4A4 H5120 / I17408,  M in 1, 2, 4, 8, 16
  decode   W4A4 H7168 / I18432,  M in 1, 8, 32, 64 (x with 1 % outliers x20)
  prefill  W4A4 H7168 / I18432,  M in 1024, 4096, 8192
  W4A16    bf16 x NVFP4, H5120 / I17408, M in 1, 16, 128, 1024
(14617 tokens per step).  A W4A4 forward is three launches:
    nvfp4_quantize(x) -> nvfp4_gemm_swiglu_quant(gate_up; SwiGLU on the fp32
    accumulators + NVFP4 requantize in the epilogue) -> nvfp4_gemm(down)
with the library choosing the kernel by M (weight-streaming tensor-core
kernels up to 64 tokens, 2-SM CTA-pair tensor-core kernels above); a W4A16
forward is bf16_fp4_gemm(gate_up) -> silu_mul_bf16 -> bf16_fp4_gemm(down).
A step is one CUDA graph holding every workload's forwards (each workload's
forwards are also captured alone, for its own replay distribution); weight
copies rotate so that the weight stream comes from HBM every step (more
copies than fit in L2).

Weights: synthetic N(0, 0.02) fp32 draws of the shared input generator
(`synth`), rounded to bf16 on the device and quantized to NVFP4 by the
library (timing does not depend on the values); x ~ N(0, 1) bf16.

Prints one JSON line (rank 0): the whole-step throughput, a roofline record
for the step's dominant kernel, and one sub-record per workload (median and
p10/p90 over >= 100 graph replays, per-M chain and GEMM times with their
roofline fractions), the elementwise kernels against HBM, an end-to-end
number through the C ABI with host copies, and the CPU oracle on a bounded
sample.  `--impl reference` times the CPU oracle instead (the slow baseline
arm).
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

# (key, synth workload id, title)
WORKLOADS = [
    ("decode_h5120", 1, "decode dense MLP W4A4 NVFP4, hidden 5120, intermediate 17408, M 1/2/4/8/16"),
    ("decode_h7168", 2, "decode dense MLP W4A4 NVFP4, DeepSeek-V3-shaped hidden 7168, intermediate 18432, "
                        "M 1/8/32/64, x with 1% outliers x20"),
    ("prefill_h7168", 3, "prefill dense MLP W4A4 NVFP4, hidden 7168, intermediate 18432, M 1024/4096/8192"),
    ("w4a16_h5120", 4, "W4A16 dense MLP (bf16 x NVFP4 weights), hidden 5120, intermediate 17408, M 1/16/128/1024"),
]
METRIC = "NVFP4 MLP tokens/s (M=1..8192 over the decode, prefill and W4A16 workloads)"
NCOPY = 4          # rotating weight copies per weight family (> L2 in total)
REPLAYS = 100      # per-workload graph replays for median / p10 / p90
REPS = 8           # back-to-back launches per per-M timing graph

# CPU oracle sample: one forward per workload at these M on 1/SLICE of the
# intermediate size (the oracle's cost is linear in I)
SLICE = 8
ORACLE_M = {1: 16, 2: 64, 3: 256, 4: 128}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--only", default=None, help="comma-separated workload keys (default: all four)")
    p.add_argument("--m", type=int, default=None, help="one batch size instead of each workload's M list")
    p.add_argument("--algo", default="auto", choices=["auto", "gemv", "tc", "tc1sm", "swapab"],
                   help="W4A4 GEMM kernel family (auto: the library's choice by M; tc: CTA pairs with 2-SM "
                        "MMAs; tc1sm: one CTA per tile)")
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


def selected(args):
    keys = args.only.split(",") if args.only else [w[0] for w in WORKLOADS]
    out = [w for w in WORKLOADS if w[0] in keys]
    if not out:
        raise SystemExit(f"--only: no workload among {keys}")
    return out


# --------------------------------------------------------------- oracle leg
class OracleSampler:
    """The CPU oracle on a bounded sample of the benchmark's workloads: one
    MLP forward per workload at ORACLE_M[wid] tokens on the first I/SLICE
    intermediate features (gate and up rows, and the matching down_proj
    input columns), same H and value recipe.  Token equivalents = M / SLICE."""

    def __init__(self, wids):
        import numpy as np
        import oracle
        import synth
        self.np, self.oracle, self.synth = np, oracle, synth
        self.w = {}
        for fam in sorted({synth.WEIGHT_SOURCE.get(w, w) for w in wids}):
            isl = synth.WORKLOADS[fam].inter // SLICE
            wgu = synth.weight(fam, "gate_up", rows=2 * isl)       # [gate slice; up slice]
            wdn = synth.weight(fam, "down", cols=isl)
            gs_gu = oracle.global_scale(np.abs(wgu).max())
            gs_dn = oracle.global_scale(np.abs(wdn).max())
            self.w[fam] = (gs_gu, oracle.quantize_nvfp4(wgu, gs_gu), gs_dn, oracle.quantize_nvfp4(wdn, gs_dn))
        self.wids = list(wids)

    def forward(self, wid):
        """One timed oracle forward of workload `wid`; returns (token
        equivalents, seconds)."""
        np, oracle, synth = self.np, self.oracle, self.synth
        m = ORACLE_M[wid]
        gs_gu, gu, gs_dn, dn = self.w[synth.WEIGHT_SOURCE.get(wid, wid)]
        _, x = synth.activations(wid, m)
        t0 = time.perf_counter()
        if synth.WORKLOADS[wid].mode == "w4a16":
            oracle.mlp_w4a16(x, gu, np.float32(1.0) / gs_gu, dn, np.float32(1.0) / gs_dn)
        else:
            gs_x = oracle.global_scale(np.abs(x).max())
            a_gu = np.float32(1.0) / (gs_x * gs_gu)
            gs_h = np.float32(448.0 * 6.0 / 8.0)
            a_dn = np.float32(1.0) / (gs_h * gs_dn)
            fwd = oracle.mlp_w4a4_fused if synth.WORKLOADS[wid].fused else oracle.mlp_w4a4_unfused
            fwd(x, gs_x, gu, a_gu, gs_h, dn, a_dn)
        return m / SLICE, time.perf_counter() - t0

    def sample(self):
        tokens, secs = 0.0, 0.0
        for wid in self.wids:
            t, s = self.forward(wid)
            tokens += t
            secs += s
        return tokens, secs

    def describe(self):
        ms = ", ".join(f"M={ORACLE_M[w]} ({self.synth.WORKLOADS[w].name})" for w in self.wids)
        return (f"CPU oracle (NumPy float64), one MLP forward per workload on the first 1/{SLICE} of the "
                f"intermediate features: {ms}; tokens counted as M/{SLICE}")

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


def run_reference(args, world, rank):
    if rank != 0:
        return
    wls = selected(args)
    smp = OracleSampler([w[1] for w in wls])
    for _ in range(args.warmup):
        smp.sample()
    tokens, secs = 0.0, 0.0
    for _ in range(args.steps):
        t, s = smp.sample()
        tokens += t
        secs += s
    value = tokens / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "; ".join(w[2] for w in wls),
                   "step": "bounded sample: " + smp.describe()},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": smp.threads(), "kind": "oracle",
                         "sample": smp.describe()},
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

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if len(r) >= 9 and num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if len(r) >= 9 and num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if len(r) >= 9 and num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            if len(r) < 9:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        loaded = [s for s, p in zip(sm, pw) if p is not None and p > 300.0] if len(pw) == len(sm) else []
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_mhz_under_load": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def pct(vals, q):
    s = sorted(vals)
    i = min(len(s) - 1, max(0, int(round(q * (len(s) - 1)))))
    return s[i]


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import nvfp4_quantized_dense_gb300 as nv
    import synth

    nv.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    pk = peaks()
    hbm_peak = pk["hbm_gbs"] if pk else 6800.0
    bf16_peak = pk["bf16_tflops"] if pk else 1900.0
    fp4_peak = bf16_peak * 6.0        # dense FP4 : dense BF16 = 13.5 : 2.25 (nominal)
    # the sustained figure (cuBLAS bf16 back to back for seconds, under the
    # power cap) is the denominator for kernels timed inside long runs of
    # back-to-back launches, as every per-M record and the step are
    bf16_sus = pk.get("bf16_tflops_sustained", bf16_peak) if pk else 1700.0
    fp4_sus = bf16_sus * 6.0
    peak_src = "measured" if pk else "fallback"
    algo = {"auto": nv.ALGO_AUTO, "gemv": nv.ALGO_GEMV, "tc": nv.ALGO_TC, "tc1sm": nv.ALGO_TC_1SM,
            "swapab": nv.ALGO_TC_SWAPAB}[args.algo]
    wls = selected(args)

    def scalar(v):
        return torch.tensor([np.float32(v)], dtype=torch.float32, device=dev)

    def gscale_np(a):
        return np.float32(np.float32(448.0 * 6.0) / np.float32(np.abs(a).max()))

    def gscale(t):
        return np.float32(np.float32(448.0 * 6.0) / np.float32(t.abs().max().float().item()))

    # ---------------------------------------------------------------- weights
    def make_weight(fam, which, layout):
        """(codes, swizzled scales, gs) of one synth weight on the device;
        layout 'interleaved' (the fused gate_up kernel's) or 'plain'."""
        w32 = synth.weight(fam, which)
        gs = gscale_np(w32)
        rows, cols = w32.shape
        wb = torch.from_numpy(w32).to(dev).to(torch.bfloat16)
        del w32
        q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        s_lin = torch.empty((rows * cols // 16,), dtype=torch.uint8, device=dev)
        nv.nvfp4_quantize(wb, rows, cols, scalar(gs), q, s_lin, nv.SF_LINEAR)
        del wb
        s = torch.empty((nv.nvfp4_sf_bytes(rows, cols),), dtype=torch.uint8, device=dev)
        if layout == "interleaved":
            qi = torch.empty_like(q)
            nv.nvfp4_prepare_gate_up_interleaved(q, s_lin, rows, cols, qi, s)
            q = qi
        else:
            nv.nvfp4_prepare_weights(q, s_lin, rows, cols, q, s)
        return q, s, gs

    need = {}     # family -> set of (which, layout)
    for _, wid, _ in wls:
        fam = synth.WEIGHT_SOURCE.get(wid, wid)
        w = synth.WORKLOADS[wid]
        st = need.setdefault(fam, set())
        st.add(("down", "plain"))
        if w.mode == "w4a16":
            st.add(("gate_up", "plain"))
        else:
            st.add(("gate_up", "interleaved"))
            if wid == 1:
                st.add(("gate_up", "plain"))      # the unfused chain (silu_mul_nvfp4_quantize)
    weights = {}     # (fam, which, layout) -> list of NCOPY (q, s, gs)
    for fam, st in need.items():
        for which, layout in sorted(st):
            base = make_weight(fam, which, layout)
            weights[(fam, which, layout)] = [base] + [(base[0].clone(), base[1].clone(), base[2])
                                                      for _ in range(NCOPY - 1)]
    torch.cuda.synchronize()
    weight_bytes = sum(c[0].numel() + c[1].numel() for v in weights.values() for c in v)

    # ------------------------------------------------------------ workloads
    SH = [None]       # the timing stream's handle (an int: no torch stream lookup per call)

    class W:
        pass

    items = []
    ws_bytes = 16
    for key, wid, title in wls:
        spec = synth.WORKLOADS[wid]
        fam = synth.WEIGHT_SOURCE.get(wid, wid)
        it = W()
        it.key, it.wid, it.title, it.spec = key, wid, title, spec
        it.hid, it.inter, it.ms = spec.hidden, spec.inter, ((args.m,) if args.m else tuple(spec.ms))
        it.w4a16 = spec.mode == "w4a16"
        it.gu = weights[(fam, "gate_up", "plain" if it.w4a16 else "interleaved")]
        it.gu_plain = weights.get((fam, "gate_up", "plain")) if wid == 1 else None
        it.dn = weights[(fam, "down", "plain")]
        mmax = max(it.ms)
        xbits, _ = synth.activations(wid, mmax)
        it.x = torch.from_numpy(xbits.view(np.int16)).to(dev).view(torch.bfloat16)
        it.gs_x = gscale(it.x)
        hid, inter = it.hid, it.inter
        # calibrate the static down_proj input scale once from one gate_up pass
        mc = min(mmax, 1024)
        gu_tmp = torch.empty((mc, 2 * inter), dtype=torch.bfloat16, device=dev)
        gq, gsf, ggs = it.gu[0]
        if it.w4a16:
            it.a_gu = scalar(np.float32(1.0) / ggs)
            it.a_dn = scalar(np.float32(1.0) / it.dn[0][2])
            it.gs_h = None
        else:
            xq = torch.empty((mc, hid // 2), dtype=torch.uint8, device=dev)
            xs = torch.empty((nv.nvfp4_sf_bytes(mc, hid),), dtype=torch.uint8, device=dev)
            nv.nvfp4_quantize(it.x[:mc].contiguous(), mc, hid, scalar(it.gs_x), xq, xs)
            it.a_gu = scalar(np.float32(1.0) / (it.gs_x * ggs))
            nv.nvfp4_gemm(xq, xs, gq, gsf, it.a_gu, gu_tmp, mc, 2 * inter, hid)
            gf = gu_tmp.float().view(mc, 2 * inter // 128, 2, 64)      # interleaved: [64 up ; 64 gate]
            u, g = gf[:, :, 0, :].reshape(mc, inter), gf[:, :, 1, :].reshape(mc, inter)
            gs_h = gscale(g * torch.sigmoid(g) * u)
            it.gs_h = scalar(gs_h)
            it.a_dn = scalar(np.float32(1.0) / (gs_h * it.dn[0][2]))
            if it.gu_plain is not None:
                it.a_gu_plain = scalar(np.float32(1.0) / (it.gs_x * it.gu_plain[0][2]))
        it.gs_x_d = scalar(it.gs_x)
        del gu_tmp
        it.out = torch.empty((sum(it.ms), hid), dtype=torch.bfloat16, device=dev)
        it.bufs = {}
        r0 = 0
        for m in it.ms:
            bf16_mid = it.w4a16 or it.gu_plain is not None    # a bf16 gate_up result is materialized
            it.bufs[m] = dict(
                x=it.x[:m], out=it.out[r0:r0 + m],
                xq=torch.empty((m, hid // 2), dtype=torch.uint8, device=dev),
                xs=torch.empty((nv.nvfp4_sf_bytes(m, hid),), dtype=torch.uint8, device=dev),
                gu=torch.empty((m, 2 * inter), dtype=torch.bfloat16, device=dev) if bf16_mid else None,
                h16=torch.empty((m, inter), dtype=torch.bfloat16, device=dev) if it.w4a16 else None,
                hq=torch.empty((m, inter // 2), dtype=torch.uint8, device=dev),
                hs=torch.empty((nv.nvfp4_sf_bytes(m, inter),), dtype=torch.uint8, device=dev))
            r0 += m
            if it.w4a16:
                ws_bytes = max(ws_bytes, nv.bf16_fp4_gemm_workspace_bytes(m, 2 * inter, hid, algo),
                               nv.bf16_fp4_gemm_workspace_bytes(m, hid, inter, algo))
            else:
                ws_bytes = max(ws_bytes, nv.nvfp4_workspace_bytes(m, 2 * inter, hid, algo),
                               nv.nvfp4_workspace_bytes(m, hid, inter, algo))
        # a second input/output set for the end-to-end run (host copies of one
        # step overlap the other step's kernels); the intermediates are shared
        it.x_alt, it.out_alt = torch.empty_like(it.x), torch.empty_like(it.out)
        alt, r0 = {}, 0
        for m in it.ms:
            alt[m] = dict(it.bufs[m], x=it.x_alt[:m], out=it.out_alt[r0:r0 + m])
            r0 += m
        it.bufsets = (it.bufs, alt)
        items.append(it)
    # one zero-filled scratch (split-K partials + arrival counters) shared by
    # every GEMM of the step: they run in stream order
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)

    def gate_up(it, m, c, s=0):
        b = it.bufsets[s][m]
        gq, gsf, _ = it.gu[c]
        if it.w4a16:
            nv.bf16_fp4_gemm_ex(b["x"], gq, gsf, it.a_gu, b["gu"], m, 2 * it.inter, it.hid, ws, ws_bytes, algo,
                                stream=SH[0])
        else:
            nv.nvfp4_gemm_swiglu_quant_ex(b["xq"], b["xs"], gq, gsf, it.a_gu, it.gs_h, b["hq"], b["hs"], m,
                                          2 * it.inter, it.hid, ws, ws_bytes, algo, stream=SH[0])

    def down(it, m, c, s=0):
        b = it.bufsets[s][m]
        dq, dsf, _ = it.dn[c]
        if it.w4a16:
            nv.bf16_fp4_gemm_ex(b["h16"], dq, dsf, it.a_dn, b["out"], m, it.hid, it.inter, ws, ws_bytes, algo,
                                stream=SH[0])
        else:
            nv.nvfp4_gemm_ex(b["hq"], b["hs"], dq, dsf, it.a_dn, b["out"], m, it.hid, it.inter, ws, ws_bytes,
                             algo, stream=SH[0])

    def forward(it, m, c, s=0):
        b = it.bufsets[s][m]
        if not it.w4a16:
            nv.nvfp4_quantize(b["x"], m, it.hid, it.gs_x_d, b["xq"], b["xs"], stream=SH[0])
        gate_up(it, m, c, s)
        if it.w4a16:
            nv.silu_mul_bf16(b["gu"], m, it.inter, b["h16"], stream=SH[0])
        down(it, m, c, s)

    def forward_unfused(it, m, c):
        """The unfused decode chain: gate_up GEMM to bf16 on the plain weight,
        then silu_mul_nvfp4_quantize, then down_proj."""
        b = it.bufs[m]
        gq, gsf, _ = it.gu_plain[c]
        nv.nvfp4_quantize(b["x"], m, it.hid, it.gs_x_d, b["xq"], b["xs"], stream=SH[0])
        nv.nvfp4_gemm_ex(b["xq"], b["xs"], gq, gsf, it.a_gu_plain, b["gu"], m, 2 * it.inter, it.hid, ws, ws_bytes,
                         algo, stream=SH[0])
        nv.silu_mul_nvfp4_quantize(b["gu"], m, it.inter, it.gs_h, b["hq"], b["hs"], stream=SH[0])
        down(it, m, c)

    def launches(it):
        """Kernels one forward of each M launches: quantize + 2 GEMMs (W4A4);
        2 GEMMs + silu_mul_bf16 (W4A16), where a tensor-core W4A16 GEMM given
        its workspace (as here, at every M) is the activation pre-pass + the
        TMEM kernel."""
        if not it.w4a16:
            return 3 * len(it.ms)
        per_gemm = 1 if algo == nv.ALGO_GEMV else 2
        return sum(2 * per_gemm + 1 for m in it.ms)

    stream = torch.cuda.Stream(device=dev)
    SH[0] = stream.cuda_stream

    def graph_of(fn):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            fn()
        return gr

    def time_graph(gr, reps=3):
        """Mean ms of one replay of `gr` over `reps` replays (after one warm)."""
        with torch.cuda.stream(stream):
            gr.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                gr.replay()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) / reps

    with torch.cuda.stream(stream):
        for it in items:                      # warm every kernel outside capture
            for m in it.ms:
                forward(it, m, 0)
        torch.cuda.synchronize()
        graphs = {it.key: [graph_of(lambda it=it, c=c: [forward(it, m, c) for m in it.ms]) for c in range(NCOPY)]
                  for it in items}
    torch.cuda.synchronize()
    tokens_per_step = sum(sum(it.ms) for it in items)
    launches_per_step = sum(launches(it) for it in items)

    # The timed step: every workload's forwards in one graph (the launches
    # stay chained by programmatic dependent launch across the workloads, as
    # they would not be across separate graph launches).
    with torch.cuda.stream(stream):
        step_graphs = [graph_of(lambda c=c: [forward(it, m, c) for it in items for m in it.ms])
                       for c in range(NCOPY)]
    torch.cuda.synchronize()

    def step(i):
        step_graphs[i % NCOPY].replay()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()

    clocks = Clocks(local)
    clocks.start()
    # ------------------------------------------------------ headline (timed)
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed_steps")       # (for profiler launch lists of exactly these steps)
    with torch.cuda.stream(stream):
        t_start.record()
        for i in range(args.steps):
            step(i)
        t_end.record()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier()
    step_ms = t_start.elapsed_time(t_end) / args.steps

    # -------------------------------------- per-workload replay distributions
    per = {}
    for it in items:
        times = []
        with torch.cuda.stream(stream):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(REPLAYS)]
            for i, (a, b) in enumerate(evs):
                a.record(stream)
                graphs[it.key][i % NCOPY].replay()
                b.record(stream)
        stream.synchronize()
        times = [a.elapsed_time(b) for a, b in evs]
        med = statistics.median(times)
        per[it.key] = {"workload": it.title, "tokens": sum(it.ms), "replays": REPLAYS,
                       "ms_median": med, "ms_p10": pct(times, 0.1), "ms_p90": pct(times, 0.9),
                       "tokens_per_s": sum(it.ms) / (med / 1000.0)}

    # --------------------- per M: whole forward and each GEMM, back to back
    def per_launch_ms(fn):
        gr = graph_of(lambda: [fn(r % NCOPY) for r in range(REPS)])
        t = time_graph(gr) / REPS
        del gr
        return t

    w_bytes = {}      # per weight tensor: codes + scales
    # the power-hungry prefill last, so that its clock drop under the power
    # cap does not carry over into the other workloads' records
    for it in [i for i in items if i.wid != 3] + [i for i in items if i.wid == 3]:
        hid, inter = it.hid, it.inter
        gu_w = 2 * inter * hid * 9 // 16
        dn_w = inter * hid * 9 // 16
        rec = per[it.key]
        rec["per_m"] = {}
        for m in it.ms:
            t_fwd = per_launch_ms(lambda c, it=it, m=m: forward(it, m, c))
            t_gu = per_launch_ms(lambda c, it=it, m=m: gate_up(it, m, c))
            t_dn = per_launch_ms(lambda c, it=it, m=m: down(it, m, c))
            r = {"forward_us": 1000 * t_fwd, "gate_up_us": 1000 * t_gu, "down_us": 1000 * t_dn,
                 "tokens_per_s": m / (t_fwd / 1000.0)}
            if it.w4a16:
                gu_b = gu_w + m * hid * 2 + m * 2 * inter * 2
                dn_b = dn_w + m * inter * 2 + m * hid * 2
                gu_f, dn_f = 2.0 * m * hid * 2 * inter, 2.0 * m * inter * hid
            else:
                gu_b = gu_w + m * hid * 9 // 16 + m * inter * 9 // 16
                dn_b = dn_w + m * inter * 9 // 16 + m * hid * 2
                gu_f, dn_f = 4.0 * m * hid * inter, 2.0 * m * inter * hid
            if m <= 64:          # weight-streaming: HBM-bound on the weight bytes
                r["gate_up_hbm_frac"] = gu_b / (t_gu / 1000) / 1e9 / hbm_peak
                r["down_hbm_frac"] = dn_b / (t_dn / 1000) / 1e9 / hbm_peak
                r["path_hbm_frac"] = (gu_w + dn_w) / (t_fwd / 1000) / 1e9 / hbm_peak
            else:                # compute-bound: tensor peak of the contraction's dtype
                pks = bf16_sus if it.w4a16 else fp4_sus
                pkb = bf16_peak if it.w4a16 else fp4_peak
                r["gate_up_tensor_frac"] = gu_f / (t_gu / 1000) / 1e12 / pks
                r["down_tensor_frac"] = dn_f / (t_dn / 1000) / 1e12 / pks
                r["gate_up_tensor_frac_of_burst"] = gu_f / (t_gu / 1000) / 1e12 / pkb
                r["down_tensor_frac_of_burst"] = dn_f / (t_dn / 1000) / 1e12 / pkb
                r["gate_up_tflops"] = gu_f / (t_gu / 1000) / 1e12
            rec["per_m"][str(m)] = r
        if it.wid == 1 and it.gu_plain is not None:
            rec["unfused_chain_forward_us"] = {
                str(m): 1000 * per_launch_ms(lambda c, it=it, m=m: forward_unfused(it, m, c)) for m in it.ms}
        w_bytes[it.key] = gu_w + dn_w

    # ------------------------------------------------- elementwise kernels
    elementwise = {}
    big = next((it for it in items if it.wid == 3), None)
    if big is not None:
        m, k = max(big.ms), big.hid
        xs2 = [big.x[:m], torch.empty_like(big.x[:m]).copy_(big.x[:m])]    # 2 x 117 MB > L2
        b = big.bufs[m]
        t = per_launch_ms(lambda c: nv.nvfp4_quantize(xs2[c % 2], m, k, big.gs_x_d, b["xq"], b["xs"],
                                                      stream=SH[0]))
        nb = m * k * 2 + m * k // 2 + m * k // 16
        elementwise["nvfp4_quantize"] = {"shape": f"[{m}, {k}]", "us": 1000 * t, "bytes": nb,
                                         "gbs": nb / (t / 1000) / 1e9, "hbm_frac": nb / (t / 1000) / 1e9 / hbm_peak}
        del xs2
    dec = next((it for it in items if it.wid in (1, 4)), None)
    if dec is not None:
        inter = dec.inter
        for m in (16, 1024):
            gus = [torch.randn((m, 2 * inter), device=dev).to(torch.bfloat16) for _ in range(2)]
            hq = torch.empty((m, inter // 2), dtype=torch.uint8, device=dev)
            hs = torch.empty((nv.nvfp4_sf_bytes(m, inter),), dtype=torch.uint8, device=dev)
            h16 = torch.empty((m, inter), dtype=torch.bfloat16, device=dev)
            gsd = scalar(64.0)
            t = per_launch_ms(lambda c: nv.silu_mul_nvfp4_quantize(gus[c % 2], m, inter, gsd, hq, hs,
                                                                   stream=SH[0]))
            nb = m * 2 * inter * 2 + m * inter // 2 + m * inter // 16
            elementwise[f"silu_mul_nvfp4_quantize_m{m}"] = {
                "shape": f"[{m}, {2 * inter}]", "us": 1000 * t, "bytes": nb, "gbs": nb / (t / 1000) / 1e9,
                "hbm_frac": nb / (t / 1000) / 1e9 / hbm_peak}
            t = per_launch_ms(lambda c: nv.silu_mul_bf16(gus[c % 2], m, inter, h16, stream=SH[0]))
            nb = m * 2 * inter * 2 + m * inter * 2
            elementwise[f"silu_mul_bf16_m{m}"] = {
                "shape": f"[{m}, {2 * inter}]", "us": 1000 * t, "bytes": nb, "gbs": nb / (t / 1000) / 1e9,
                "hbm_frac": nb / (t / 1000) / 1e9 / hbm_peak}
            del gus
    clk = clocks.stop()

    step_ms, value = aggregate(step_ms, tokens_per_step, world, device=dev)

    # roofline of the step's dominant kernel: the GEMM with the largest share
    # of the step time
    dom = None
    for it in items:
        for m in it.ms:
            r = per[it.key]["per_m"][str(m)]
            for which in ("gate_up", "down"):
                t = r[f"{which}_us"]
                if dom is None or t > dom[0]:
                    dom = (t, it, m, which)
    # DRAM bytes (read + write) per launch of the step's GEMMs from an ncu
    # capture of this bench's own timed step (default workloads, one pass per
    # launch): reported as the roofline's traffic when that launch is the
    # dominant one; to be removed whenever the kernel changes before it is
    # captured again
    measured_traffic = {("prefill_h7168", 8192, "gate_up"): 287.8e6,
                        ("prefill_h7168", 8192, "down"): 523.2e6}
    roofline = None
    if dom is not None:
        t_us, it, m, which = dom
        r = per[it.key]["per_m"][str(m)]
        if m > 64:
            flops = (4.0 if which == "gate_up" else 2.0) * m * it.hid * it.inter
            pkk = bf16_sus if it.w4a16 else fp4_sus
            pkb = bf16_peak if it.w4a16 else fp4_peak
            achieved = flops / (t_us / 1e6) / 1e12
            roofline = {"bound": "tensor", "achieved": achieved, "peak": pkk, "unit": "TFLOP/s",
                        "frac": achieved / pkk, "traffic": None,
                        "algorithmic_flops_per_launch": flops,
                        "peak_note": ("measured bf16 sustained" if it.w4a16 else
                                      "measured bf16 sustained x 6 (nominal fp4 : bf16)") + f" ({peak_src}); "
                                     "the kernel is timed inside runs of back-to-back launches",
                        "peak_burst": pkb, "frac_of_burst": achieved / pkb}
        else:
            nb = r[f"{which}_hbm_frac"] * hbm_peak * 1e9 * (t_us / 1e6)
            achieved = nb / (t_us / 1e6) / 1e9
            roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                        "frac": achieved / hbm_peak, "traffic": None, "algorithmic_bytes_per_launch": nb,
                        "peak_note": f"measured copy bandwidth ({peak_src})"}
        fused = not it.w4a16 and which == "gate_up"
        roofline["kernel"] = (f"{'nvfp4_gemm_swiglu_quant' if fused else ('bf16_fp4_gemm' if it.w4a16 else 'nvfp4_gemm')} "
                              f"{which} ({it.key}, M={m})")
        roofline["us_per_launch"] = t_us
        roofline["traffic"] = measured_traffic.get((it.key, m, which))
        if roofline["traffic"] is not None:
            roofline["traffic_unit"] = "DRAM bytes read + written per launch (ncu, the bench's timed step)"
        roofline["timing"] = (f"{REPS} launches back to back in one CUDA graph (weight copies rotating), CUDA "
                              "events on the launching stream around 3 replays")

    # ------------------------------------------- end to end through the C ABI
    x_host = {it.key: it.x.cpu().pin_memory() for it in items}
    out_host = {it.key: torch.empty(it.out.shape, dtype=torch.bfloat16).pin_memory() for it in items}
    h2d = sum(it.x.numel() * 2 for it in items)
    d2h = sum(it.out.numel() * 2 for it in items)
    e2e_steps = max(3, min(args.steps, 20))
    # Every step copies every workload's x in from pinned host memory and its
    # output back out, on two streams of their own (one per direction).  The
    # steps alternate between two device input/output sets, so that the copies
    # of one step run under the kernels of its neighbours: step i's inputs go
    # in once step i-2 (the same set) has read them, its kernels (the step's
    # graph, as in the timed arm) wait for those inputs and for step i-2's
    # outputs to have left, and its outputs go out as soon as it is done.
    with torch.cuda.stream(stream):
        e2e_graphs = [[graph_of(lambda c=c, s=s: [forward(it, m, c, s) for it in items for m in it.ms])
                       for c in range(NCOPY)] for s in range(2)]
    torch.cuda.synchronize()
    in_stream, out_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    order = sorted(items, key=lambda it: -(it.x.numel() + it.out.numel()))

    def copy_gbs(dst, src, stream_):
        """This machine's host-link rate for one copy of the step's size (the
        end-to-end number is bound by it where it is slow)."""
        with torch.cuda.stream(stream_):
            dst.copy_(src, non_blocking=True)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream_)
            for _ in range(3):
                dst.copy_(src, non_blocking=True)
            e1.record(stream_)
        stream_.synchronize()
        return src.numel() * src.element_size() * 3 / (e0.elapsed_time(e1) / 1e3) / 1e9

    big = order[0]
    link = {"h2d_gbs": copy_gbs(big.x, x_host[big.key], in_stream),
            "d2h_gbs": copy_gbs(out_host[big.key], big.out, out_stream)}
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for st in range(2):                         # (so that the first waits are satisfied)
        ev_done[st].record(stream)
        ev_out[st].record(out_stream)
    torch.cuda.synchronize()

    def e2e_step(i):
        st = i % 2
        in_stream.wait_event(ev_done[st])
        with torch.cuda.stream(in_stream):
            for it in order:
                (it.x, it.x_alt)[st].copy_(x_host[it.key], non_blocking=True)
        ev_in[st].record(in_stream)
        stream.wait_event(ev_in[st])
        stream.wait_event(ev_out[st])
        with torch.cuda.stream(stream):
            e2e_graphs[st][i % NCOPY].replay()
        ev_done[st].record(stream)
        out_stream.wait_event(ev_done[st])
        with torch.cuda.stream(out_stream):
            for it in order:
                out_host[it.key].copy_((it.out, it.out_alt)[st], non_blocking=True)
        ev_out[st].record(out_stream)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - w0) / e2e_steps
    e2e_value = world * tokens_per_step / e2e_s
    del e2e_graphs

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        smp = OracleSampler([it.wid for it in items])
        tokens, secs = 0.0, 0.0
        for _ in range(2):
            t, s = smp.sample()
            tokens += t
            secs += s
        cpu = {"value": tokens / secs, "unit": "tokens/s", "cores": smp.threads(), "kind": "oracle",
               "sample": smp.describe() + "; two passes"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "nvfp4 (e2m1 x ue4m3, fp32 accumulate); bf16 x nvfp4 in the W4A16 workload",
            "data": "synthetic",
            "config": {"workload": "; ".join(it.title for it in items), "tokens_per_step": tokens_per_step,
                       "step": "one MLP forward per (workload, M), all in one CUDA graph per step",
                       "l2": f"{NCOPY} rotating weight copies per weight family, {weight_bytes / 1e6:.0f} MB > L2",
                       "weights": "synth N(0, 0.02) fp32 draws, rounded to bf16 and quantized to NVFP4 on the "
                                  "device by the library",
                       "parallelism": f"replicas{world}", **({"algo": args.algo} if args.algo != "auto" else {})},
            "roofline": roofline, "per_workload": per, "elementwise": elementwise,
            "cpu_baseline": cpu, "clocks": clk,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "host_link": link,
                    "note": "host wall clock per step; pinned host buffers; x of every workload in and every "
                            "output out, each step, on two copy streams of their own; the steps alternate "
                            "between two device input/output sets so that one step's copies overlap its "
                            "neighbours' kernels; the step's API calls replayed from their CUDA graph"},
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
