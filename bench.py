"""Benchmark of the routed block-scaled MoE layer on GB300.

One step = one moe_forward over one seeded token batch (router, dispatch,
activation quantisation, GEMM1 + capped SwiGLU, h quantisation, GEMM2,
combine), inputs resident in HBM.  Prints one JSON line.  The line's workload
is the largest single-GPU configuration (a 16384-token MXFP8 prefill chunk
with Zipf-skewed expert load); the other configurations (the tiny case, the
1-, 8-, 32-, 64- and 192-token decode batches, the 4096-token NVFP4 prefill
chunk) are measured in the same run under `per_workload`.  The tensor-core roofs are the
block-scaled MMA rates measured in the same run (moe_bench_mma_peak).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Multi-GPU: token-sharded replicas (each rank runs its own batch and holds all
experts; no collective on the data path); value = all ranks' tokens / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("MoE-layer tokens/s & µs/layer; % HBM roofline (decode) / % FP4-FP8 peak (prefill)")
DEFAULT_WORKLOAD = "prefill16384_mxfp8_zipf"
# the other configurations, measured beside the line's (timed steps, CPU work
# kept small): name -> steps
PER_WORKLOAD = {"tiny_mxfp8": 2000, "decode1_nvfp4": 2000, "decode8_nvfp4": 1000, "decode32_mxfp8": 500,
                "decode64_nvfp4": 1000, "decode192_mxfp8_outliers": 500, "prefill4096_nvfp4": 200}
UNIT = "tokens/s"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_traffic.json")


# dense tensor-core peak per dtype relative to bf16 (nominal GB300 figures:
# 2.25 PFLOP/s bf16, 4.5 fp8, 13.5 fp4); used only if the measurement of the
# block-scaled MMA rate is switched off
TENSOR_RATIO = {"nvfp4": 13.5 / 2.25, "mxfp8": 4.5 / 2.25}


def peaks():
    """HBM copy bandwidth and the sustained bf16 GEMM rate (the GEMMs are timed
    inside a long step): measured on this GPU type, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1700.0, source="fallback")


def kernel_source_sha() -> str:
    """Hash of the expert-GEMM sources (the traffic figures in profiles/ hold
    only for the kernels they were captured from)."""
    h = hashlib.sha256()
    for f in ("moe_gemm.cu", "moe_gemm_common.cuh", "moe_ffn_decode.cu", "moe_common.cuh", "moe_quant_dev.cuh"):
        h.update(open(os.path.join(ROOT, "block_scaled_fp4_route_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_key(kname: str, w: dict, tile_rows: int) -> str:
    """Which measured kernel a roof's traffic ratio comes from."""
    if kname == "ffn":
        return f"ffn_decode_{w['fmt']}"
    return f"{kname}_{'token_major' if tile_rows == 128 else 'decode'}_{w['fmt']}"


def write_traffic(pairs):
    """profiles/gemm_traffic.json from ncu captures of small cases: each pair
    is (the plain bench run's JSON line, the ncu CSV of dram__bytes_read.sum
    and dram__bytes_write.sum of its GEMM launches).  Per kernel, the mean
    DRAM bytes per launch over its algorithmic bytes (kernel_bytes) is stored
    with the GEMM sources' hash; the bench applies the ratio to a full
    workload's algorithmic bytes (traffic grows with the units processed:
    touched experts' weights, pairs' activations)."""
    import csv
    import synth
    out = {"source_sha": kernel_source_sha(),
           "how": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum per launch on small cases; ratio = "
                  "mean DRAM bytes per launch / algorithmic bytes (bench.py kernel_bytes); the bench multiplies a "
                  "full workload's algorithmic bytes by the ratio",
           "ratios": {}}
    for js, cs in pairs:
        line = json.loads(open(js).read().strip().splitlines()[-1])
        cfg = line["config"]
        w = dict(synth.WORKLOADS[cfg["workload"]])
        fused = cfg["ffn_schedule"] == "fused decode kernel"
        kb = kernel_bytes(w, cfg["touched_experts"], fused, cfg.get("y_format", "fp16e") == "fp16e")
        per = {}
        rows = list(csv.reader(l for l in open(cs) if l.startswith('"')))
        hdr = rows[0]
        ki, ii, mi, vi = (hdr.index(n) for n in ("Kernel Name", "ID", "Metric Name", "Metric Value"))
        for r in rows[1:]:
            if r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
                continue
            per.setdefault((r[ki], r[ii]), 0.0)
            per[(r[ki], r[ii])] += float(r[vi].replace(",", ""))
        groups = {}
        for (kn, _), b in per.items():
            kname = "ffn" if "k_moe_ffn_decode" in kn else ("gemm1" if kn.split("(")[0].endswith("1>") else "gemm2")
            groups.setdefault(kname, []).append(b)
        for kname, vals in groups.items():
            mean = sum(vals) / len(vals)
            key = traffic_key(kname, w, cfg.get("tile_rows", 128 if not fused else 64))
            out["ratios"][key] = {"workload": cfg["workload"], "launches": len(vals), "dram_bytes": mean,
                                  "algorithmic_bytes": kb[kname], "ratio": round(mean / kb[kname], 4)}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps(out, indent=1))


# ----------------------------------------------------------------------------
# algorithmic bytes of one launch of each expert GEMM
# ----------------------------------------------------------------------------

def gemm_bytes(w: dict, n_touched: int, h_quantised_in_gemm1: bool = False, y_compact: bool = True):
    """Algorithmic HBM bytes of GEMM1 (gate+up) and GEMM2 (down) per launch:
    the encoded weights of the touched experts (each read once), the encoded
    activations read and the output written (GEMM1: bf16 h, or its MXFP8
    codes and scales when the epilogue quantises h; GEMM2: y rows, fp16 codes
    plus an exponent byte per 32 features, or fp32)."""
    H, F, P = w["H"], w["F"], w["T"] * w["k"]
    nv = w["fmt"] == "nvfp4"
    bpe = 0.5 + 1 / 16 if nv else 1 + 1 / 32          # bytes per element incl. block scales
    glob = 4 if nv else 0
    h_out = P * F * (bpe if h_quantised_in_gemm1 else 2)
    g1 = n_touched * (2 * (F * H * bpe + glob)) + P * (H * bpe + glob) + h_out
    g2 = n_touched * (H * F * bpe + glob) + P * (F * bpe + glob) + P * H * (2 + 1 / 32 if y_compact else 4)
    return g1, g2


def kernel_bytes(w: dict, n_touched: int, fused: bool, y_compact: bool = True) -> dict:
    """Algorithmic bytes per launch of the kernels whose roofs the bench
    reports: gemm1 and gemm2 (separate kernels; GEMM1 writes MXFP8 h codes in
    its epilogue, NVFP4 h as bf16), or ffn (the fused decode kernel: both
    GEMMs' bytes without the h round trip, which stays in L2)."""
    mx = w["fmt"] == "mxfp8"
    g1, g2 = gemm_bytes(w, n_touched, mx, y_compact)
    if not fused:
        return {"gemm1": g1, "gemm2": g2}
    P, F = w["T"] * w["k"], w["F"]
    bpe = 1 + 1 / 32 if mx else 0.5 + 1 / 16
    h_write = P * F * (bpe if mx else 2)             # GEMM1's h out (MXFP8 codes + scales, or bf16)
    h_read = P * (F * bpe + (0 if mx else 4))        # GEMM2's encoded h in
    return {"ffn": g1 + g2 - h_write - h_read}


def gemm_flops(w: dict):
    """Useful flops of GEMM1 (gate and up: 2 x 2 H F per pair) and GEMM2 (2 H F per pair)."""
    P = w["T"] * w["k"]
    return 4.0 * P * w["H"] * w["F"], 2.0 * P * w["H"] * w["F"]


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.window = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                       "-lms", "100", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.p.stdout:
            self.samples.append((time.time(), [s.strip() for s in line.split(",")]))

    def start(self):
        self.window = [time.time(), None]

    def stop(self):
        self.window[1] = time.time()
        if self.p:
            time.sleep(0.25)
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()

    def summary(self):
        if not self.p:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        t0, t1 = self.window
        rows = [r for (t, r) in self.samples if t0 <= t <= t1 + 0.1]
        if not rows:   # timed region shorter than the sampling period: nearest samples
            rows = [r for (t, r) in self.samples if t0 - 0.3 <= t <= t1 + 0.3]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------------------
# replicas across ranks: no collective on the data path, only the timing
# ----------------------------------------------------------------------------

def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The slowest rank's time (every rank gets the same number)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank_step: int, steps: int, world: int, slowest_ms: float) -> float:
    """Whole-job throughput: the tokens of every rank over the slowest rank's time."""
    return world * tokens_per_rank_step * steps / (slowest_ms / 1e3)


# ----------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)
# ----------------------------------------------------------------------------

class OracleSample:
    """The oracle as it stands on a bounded sample of a workload: given the
    inputs and the encoded experts (prepared outside the timing), one call
    routes the sample tokens, dispatches them, runs every (token, expert) pair
    through the quantised FFN (weights decoded on the fly) and combines."""

    def __init__(self, w: dict, n_tokens: int, max_pairs=None):
        import oracle
        import synth
        self.oracle, self.w = oracle, w
        rng = np.random.default_rng(77)
        self.tokens = np.sort(rng.choice(w["T"], size=min(n_tokens, w["T"]), replace=False))
        self.inputs = (synth.x_rows(w, self.tokens), synth.router_weight(w), synth.router_bias(w))
        self.max_pairs = max_pairs
        res = oracle.route(self.inputs[0], self.inputs[1], self.inputs[2], w["k"])
        order = oracle.dispatch(res["idx"], w["E"])
        P = len(self.tokens) * w["k"] if max_pairs is None else max_pairs
        experts = sorted(set(int(e) for e in res["idx"].ravel()[order["perm"][:P]]))
        self.cache = {e: oracle.quantized_expert(w, e) for e in experts}
        self.pairs = P

    def run(self):
        return self.oracle.moe_layer(self.w, self.tokens, inputs=self.inputs, expert_cache=self.cache,
                                     max_pairs=self.max_pairs)

    def tokens_per_call(self) -> float:
        return self.pairs / self.w["k"]


def cpu_cores() -> int:
    import oracle
    return oracle.num_threads()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import synth
    w = synth.WORKLOADS[args.workload]
    # size one step so that warmup + steps take about two minutes of CPU
    probe = OracleSample(w, 1, max_pairs=1)
    t0 = time.perf_counter()
    probe.run()
    t_pair = time.perf_counter() - t0
    n_pairs = int(max(1, min(w["k"], 120.0 / max(1, args.steps + args.warmup) / max(t_pair, 1e-6))))
    samp = OracleSample(w, 1, max_pairs=n_pairs)
    for _ in range(args.warmup):
        samp.run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        samp.run()
    dt = time.perf_counter() - t0
    value = samp.tokens_per_call() * args.steps / dt
    cores = cpu_cores()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload, **{k: w[k] for k in ("T", "H", "E", "k", "F", "fmt")}},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"per step: routing of 1 token of {args.workload} and {n_pairs} of its "
                                       f"{w['k']} expert FFN pairs (weights decoded in fp64), counted as "
                                       f"{n_pairs}/{w['k']} token"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# measured block-scaled tensor-core rates (moe_bench_mma_peak)
# ----------------------------------------------------------------------------

def measure_tensor_peaks(moe, torch, gpu_index: int, burst_s: float = 0.1, sustained_s: float = 2.0):
    """Dense block-scaled MMA rate of this GPU per format, measured with the
    same MMA forms the expert GEMMs issue (one CTA per SM, operands on chip,
    no HBM traffic): `burst` = one launch of ~burst_s after a warm-up launch,
    `sustained` = back-to-back launches for ~sustained_s (the power cap's
    steady state, the right denominator for a kernel timed inside a long
    step), each with the SM clock sampled while it ran."""
    out = {}
    st = torch.cuda.current_stream()
    status = torch.zeros(64, dtype=torch.int32, device="cuda")
    for fmt in ("nvfp4", "mxfp8"):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

        def timed(n, reps):
            ev[0].record(st)
            for _ in range(reps):
                ctas, fpm = moe.moe_bench_mma_peak(fmt, n, status)
            ev[1].record(st)
            torch.cuda.synchronize()
            if moe.moe_poll_device_status(status) != 0:
                raise RuntimeError(f"tensor-core peak kernel ({fmt}): a bounded wait ran out")
            return ev[0].elapsed_time(ev[1]) * 1e-3, ctas, fpm

        n = 1 << 14
        t, ctas, fpm = timed(n, 1)
        n = max(4, int(n * burst_s / max(t, 1e-6)) // 4 * 4)
        timed(n, 1)                                   # warm-up at the burst length
        clk = ClockSampler(gpu_index)
        time.sleep(0.3)
        clk.start()
        tb, ctas, fpm = timed(n, 1)
        clk.stop()
        burst = {"tflops": ctas * n * fpm / tb / 1e12, "seconds": tb, "clocks": clk.summary()}
        reps = max(1, int(round(sustained_s / tb)))
        clk = ClockSampler(gpu_index)
        time.sleep(0.3)
        clk.start()
        ts, ctas, fpm = timed(n, reps)
        clk.stop()
        sus = {"tflops": ctas * n * fpm * reps / ts / 1e12, "seconds": ts, "clocks": clk.summary()}
        out[fmt] = {"burst": burst, "sustained": sus, "ctas": ctas, "mmas_per_cta": n, "flops_per_mma": fpm,
                    "mma": "tcgen05 M=128 N=256 K=%d %s" % (64 if fmt == "nvfp4" else 32,
                                                          "kind::mxf4nvf4 scale_vec::4X" if fmt == "nvfp4"
                                                          else "kind::mxf8f6f4 scale_vec::1X")}
    return out


# ----------------------------------------------------------------------------
# the MXFP8 KV-cache quantiser (moe_kv_quantize_mxfp8)
# ----------------------------------------------------------------------------

def measure_kv_quant(moe, torch, hbm_gbs: float, tokens=16384, heads=8, head_dim=128, reps=50):
    """New K rows of a prefill chunk, bf16 [tokens, heads, head_dim], encoded
    into a paged cache twice their size at a seeded permutation of slots:
    algorithmic bytes = 2 (bf16 in) + 1 + 1/32 (codes and E8M0 scales out) per
    element; the inputs (34 MB in, 17 MB out) fit in L2, so an L2 flush
    buffer is written between the timed launches."""
    g = torch.Generator(device="cuda").manual_seed(5)
    kv = torch.randn((tokens, heads, head_dim), device="cuda", generator=g).to(torch.bfloat16)
    slots = torch.randperm(2 * tokens, device="cuda", generator=g)[:tokens].to(torch.int64)
    codes = torch.empty((2 * tokens, heads, head_dim), dtype=torch.uint8, device="cuda")
    scales = torch.empty((2 * tokens, heads, head_dim // 32), dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    for _ in range(3):
        moe.moe_kv_quantize_mxfp8(kv, codes, scales, slots=slots)
    times = []
    for _ in range(reps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        moe.moe_kv_quantize_mxfp8(kv, codes, scales, slots=slots)
        b.record(st)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e-3)
    sec = float(np.median(times))
    n = tokens * heads * head_dim
    alg = n * (2 + 1 + 1 / 32)
    return {"tokens": tokens, "heads": heads, "head_dim": head_dim, "slot_map": "seeded permutation into 2x slots",
            "us": sec * 1e6, "gbs": alg / sec / 1e9, "hbm_frac": alg / sec / 1e9 / hbm_gbs,
            "algorithmic_bytes": alg, "l2": "256 MB flush buffer written before each timed launch", "reps": reps}


# ----------------------------------------------------------------------------
# one workload on the GPU
# ----------------------------------------------------------------------------

def capture_graph(torch, gw, G: int):
    """G moe_forward calls captured in one CUDA graph (a serving loop's
    decode step); each captured call reads its inputs on every replay."""
    st = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(st)
    with torch.cuda.stream(side):
        gw.forward()
    st.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(G):
            gw.forward()
    graph.replay()
    torch.cuda.synchronize()
    return graph


def stage_times(moe, torch, gw, n: int) -> dict:
    """Mean device time of each stage (events between the stages of
    moe_forward_profiled, same stream) over n calls."""
    st = torch.cuda.current_stream()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.NUM_STAGES + 1)] for _ in range(n)]
    for row in evs:          # torch creates the CUDA event on its first record
        for e in row:
            e.record(st)
    for i in range(n):
        moe.moe_forward_profiled(gw.cfg, gw.x, gw.w_router, gw.bias, gw.qw["gate"], gw.qw["up"], gw.qw["down"],
                                 gw.out, gw.ws, evs[i])
    torch.cuda.synchronize()
    return {nm: float(np.mean([e[i].elapsed_time(e[i + 1]) for e in evs])) for i, nm in enumerate(moe.STAGE_NAMES)}


def ffn_fused(gw) -> bool:
    """Whether this configuration runs GEMM1, the h quantisation and GEMM2 as
    the fused decode kernel (the library decides: its forward then launches
    fewer kernels than with ffn_schedule = 1)."""
    moe = gw.moe
    c = gw.cfg
    sep = moe.make_config(c.T, c.H, c.E, c.k, c.F, c.fmt, c.swiglu_cap, c.mx_scale_mode, c.bias_in_weights,
                          c.routed_scale, c.act_global_mode, ffn_schedule=1, y_format=c.y_format)
    return moe.moe_forward_kernel_count(c) < moe.moe_forward_kernel_count(sep)


def rooflines(w: dict, gw, n_touched: int, ms_per_step: float, stage_ms: dict, hbm_gbs: float, tpeak: float):
    """Roofline fractions of GEMM1, GEMM2 and the whole layer: algorithmic
    bytes over the HBM copy bandwidth and useful flops over the dtype's
    tensor-core rate (tpeak, TFLOP/s); `bound` is the roof that binds by
    arithmetic intensity.  Where one fused kernel runs both GEMMs (decode
    batches) its roof ("ffn") counts the bytes and flops of both and the
    separate GEMM entries are absent.  The layer's algorithmic bytes are the
    touched experts' encoded weights, the router weights, x and the output:
    the intermediates (x codes, h, y) are the implementation's traffic, which
    one fused kernel per layer could keep on chip; each GEMM's own roof counts
    the activations it reads and writes."""
    fused = ffn_fused(gw)
    kb = kernel_bytes(w, n_touched, fused, gw.cfg.y_format == gw.moe.Y_FP16E)
    g1_flops, g2_flops = gemm_flops(w)
    g1_s, g2_s = stage_ms["gemm1_gate_up_swiglu"] / 1e3, stage_ms["gemm2_down"] / 1e3
    balance = tpeak * 1e12 / (hbm_gbs * 1e9)        # flop per byte at which the two roofs meet
    T, H = w["T"], w["H"]
    nv = w["fmt"] == "nvfp4"
    per_expert = 3 * (w["F"] * H * (0.5 + 1 / 16 if nv else 1 + 1 / 32) + (4 if nv else 0))
    layer_bytes = n_touched * per_expert + w["E"] * H * 2 + T * H * 4
    layer_flops = g1_flops + g2_flops + 2.0 * T * H * w["E"]
    step_s = ms_per_step / 1e3

    def roof(b, f, sec):
        tensor_bound = f / b > balance
        return {"bound": "tensor" if tensor_bound else "hbm", "hbm_frac": b / sec / 1e9 / hbm_gbs,
                "tensor_frac": f / sec / 1e12 / tpeak, "gbs": b / sec / 1e9, "tflops": f / sec / 1e12,
                "frac": (f / sec / 1e12 / tpeak) if tensor_bound else (b / sec / 1e9 / hbm_gbs),
                "algorithmic_bytes": b, "flops": f}

    if fused:
        ffn = roof(kb["ffn"], g1_flops + g2_flops, g1_s)
        return {"ffn": ffn, "layer": roof(layer_bytes, layer_flops, step_s), "machine_balance_flop_per_byte": balance}
    return {"gemm1": roof(kb["gemm1"], g1_flops, g1_s), "gemm2": roof(kb["gemm2"], g2_flops, g2_s),
            "layer": roof(layer_bytes, layer_flops, step_s), "machine_balance_flop_per_byte": balance}


def measure_workload(moe, torch, name: str, steps: int, warmup: int, launch: str, tensor_peaks: dict, hbm_gbs: float,
                     gpu_index: int, dist=None, world: int = 1, n_prof: int = 200, ffn_schedule: int = 0,
                     y_format: str = "fp16e"):
    """Set up one seeded workload, time `steps` forwards (CUDA-graph replays
    of captured calls, or eager calls) between events on the launching
    stream, with the SM clock sampled, plus per-stage event times."""
    import synth
    from synth.gpu_workload import GpuWorkload
    w = synth.WORKLOADS[name]
    gw = GpuWorkload(name, torch, ffn_schedule=ffn_schedule, y_format=y_format)
    st = torch.cuda.current_stream()
    for _ in range(warmup):
        gw.forward()
    torch.cuda.synchronize()
    status = moe.moe_poll_device_status(gw.ws)
    if status != 0:
        raise RuntimeError(f"{name}: device status {status} after warmup")
    n_touched = int((gw.routing()["counts"] > 0).sum())
    G = max(d for d in range(1, 21) if steps % d == 0)
    graph = None
    if launch == "graph":
        graph = capture_graph(torch, gw, G)
        status = moe.moe_poll_device_status(gw.ws)
        if status != 0:
            raise RuntimeError(f"{name}: device status {status} after the graph warm-up replay")
        how = f"cuda_graph: {G} moe_forward calls per graph, {steps // G} replays"
    else:
        how = "eager: one moe_forward call per step"
    clocks = ClockSampler(gpu_index)
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    start.record(st)
    if graph is not None:
        for _ in range(steps // G):
            graph.replay()
    else:
        for _ in range(steps):
            gw.forward()
    end.record(st)
    torch.cuda.synchronize()
    clocks.stop()
    if dist:
        dist.barrier()
    ms = max_over_ranks(start.elapsed_time(end), dist, "cuda")
    status = moe.moe_poll_device_status(gw.ws)
    if status != 0:
        raise RuntimeError(f"{name}: device status {status} after the timed steps")
    del graph
    ms_per_step = ms / steps
    stage_ms = stage_times(moe, torch, gw, min(steps, n_prof))
    tpk = tensor_peaks[w["fmt"]]
    roof = rooflines(w, gw, n_touched, ms_per_step, stage_ms, hbm_gbs, tpk)
    if ffn_fused(gw):   # one kernel between the x quantisation and the combine
        ffn_ms = stage_ms.pop("gemm1_gate_up_swiglu") + stage_ms.pop("quant_h") + stage_ms.pop("gemm2_down")
        stage_ms = {"router": stage_ms["router"], "dispatch": stage_ms["dispatch"], "quant_x": stage_ms["quant_x"],
                    "expert_ffn_fused": ffn_ms, "combine": stage_ms["combine"]}
    res = {"workload": name, "T": w["T"], "fmt": w["fmt"], "touched_experts": n_touched, "steps": steps,
           "launch": how, "ffn_schedule": "fused decode kernel" if ffn_fused(gw) else "separate kernels",
           "y_format": y_format, "tile_rows": int(gw.layout["tile_rows"]), "ms_per_step": ms_per_step,
           "us_per_layer": ms_per_step * 1e3,
           "tokens_per_s": job_tokens_per_s(w["T"], steps, world, ms), "stage_ms": stage_ms,
           "roofline": roof, "clocks": clocks.summary(),
           "gpu_launches": moe.moe_forward_kernel_count(gw.cfg) * steps}
    return gw, res


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true", help="skip the other configurations")
    ap.add_argument("--no-tensor-peak", action="store_true",
                    help="skip the MMA-rate measurement (tensor roofs from the bf16 rate x nominal ratio)")
    ap.add_argument("--write-traffic", nargs="+", metavar="JSON,CSV",
                    help="write profiles/gemm_traffic.json from plain-run JSON lines and their ncu DRAM-byte CSVs "
                         "(no GPU needed), then exit")
    ap.add_argument("--y-format", default="fp16e", choices=["fp16e", "fp32"],
                    help="moe_config.y_format: the expert outputs between the down GEMM and the combine as fp16 "
                         "codes with an exponent per 32 features (default) or fp32")
    ap.add_argument("--ffn-schedule", type=int, default=0, choices=[0, 1],
                    help="moe_config.ffn_schedule: 0 = decode batches run the expert FFN as one fused kernel, "
                         "1 = separate kernels")
    ap.add_argument("--launch", default="graph", choices=["graph", "eager"],
                    help="timed steps as CUDA-graph replays of captured moe_forward calls (default) or eager calls")
    args = ap.parse_args()
    if args.write_traffic:
        write_traffic([tuple(p.split(",")) for p in args.write_traffic])
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch

    import block_scaled_fp4_route_gb300 as moe
    import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    gpu_index = int(vis.split(",")[local]) if vis else local

    pk = peaks()
    # ---- the tensor-core roofs: measured block-scaled MMA rates ----
    if args.no_tensor_peak:
        mma = None
        tpeak = {f: pk["bf16_tflops"] * TENSOR_RATIO[f] for f in TENSOR_RATIO}
        tsrc = f"sustained bf16 ({pk['source']}) x nominal dtype ratio"
    else:
        mma = measure_tensor_peaks(moe, torch, gpu_index)
        # the GEMMs are timed inside a long run of steps: the sustained rate
        tpeak = {f: mma[f]["sustained"]["tflops"] for f in mma}
        tsrc = "measured_tcgen05"

    w = synth.WORKLOADS[args.workload]
    T, k = w["T"], w["k"]
    gw, main_res = measure_workload(moe, torch, args.workload, args.steps, args.warmup, args.launch, tpeak,
                                    pk["hbm_gbs"], gpu_index, dist, world, ffn_schedule=args.ffn_schedule,
                                    y_format=args.y_format)
    st = torch.cuda.current_stream()
    ms_per_step = main_res["ms_per_step"]
    value = main_res["tokens_per_s"]

    # ---- distribution of single eager steps (an event between consecutive
    # calls; the timed region above gives `value`) ----
    n_dist = min(args.steps, 200)
    sev = [torch.cuda.Event(enable_timing=True) for _ in range(n_dist + 1)]
    sev[0].record(st)
    for i in range(n_dist):
        gw.forward()
        sev[i + 1].record(st)
    torch.cuda.synchronize()
    step_us = np.array([sev[i].elapsed_time(sev[i + 1]) * 1e3 for i in range(n_dist)])
    step_dist = {"steps": n_dist, "launch": "eager", "median": float(np.median(step_us)),
                 "p10": float(np.percentile(step_us, 10)), "p90": float(np.percentile(step_us, 90))}

    # ---- end to end through host buffers ----
    # Every step copies its x from pinned host memory and reads its output
    # back into a host buffer of its own, through the public moe_forward.  The
    # steps are pipelined as a serving loop would run them: two device buffer
    # sets, the copies on their own streams, ordered by events, so step i+1's
    # input copy and step i-1's output copy overlap step i's layer; the host
    # waits once, after the last step.
    e2e = None
    if not args.no_e2e:
        n_e2e = min(args.steps, 500)
        x_host = gw.x.cpu().pin_memory()
        out_host = [torch.empty_like(gw.out, device="cpu").pin_memory() for _ in range(2)]
        x_dev = [torch.empty_like(gw.x) for _ in range(2)]
        out_dev = [torch.empty_like(gw.out) for _ in range(2)]
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        ev_h2d = [torch.cuda.Event() for _ in range(2)]
        ev_fwd = [torch.cuda.Event() for _ in range(2)]
        ev_d2h = [torch.cuda.Event() for _ in range(2)]
        for b in range(2):  # every event recorded once before it is waited on
            ev_fwd[b].record(st)
            ev_d2h[b].record(st)

        def e2e_step(i):
            b = i & 1
            with torch.cuda.stream(h2d):
                h2d.wait_event(ev_fwd[b])              # step i-2 is done with x_dev[b]
                x_dev[b].copy_(x_host, non_blocking=True)
                ev_h2d[b].record(h2d)
            st.wait_event(ev_h2d[b])
            st.wait_event(ev_d2h[b])                   # step i-2's output has left out_dev[b]
            moe.moe_forward(gw.cfg, x_dev[b], gw.w_router, gw.bias, gw.qw["gate"], gw.qw["up"],
                            gw.qw["down"], out_dev[b], gw.ws)
            ev_fwd[b].record(st)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_fwd[b])
                out_host[b].copy_(out_dev[b], non_blocking=True)
                ev_d2h[b].record(d2h)

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        t0 = time.perf_counter()
        for i in range(n_e2e):
            e2e_step(i)
        torch.cuda.synchronize()
        dt = max_over_ranks(time.perf_counter() - t0, dist, "cuda")
        assert torch.equal(out_host[(n_e2e - 1) & 1].view(torch.int16), gw.out.cpu().view(torch.int16)), \
            "end-to-end output differs from the device-resident run"
        e2e = {"value": job_tokens_per_s(T, n_e2e, world, dt * 1e3), "unit": UNIT,
               "h2d_bytes_per_step": int(gw.x.numel() * 2), "d2h_bytes_per_step": int(gw.out.numel() * 2),
               "steps": n_e2e,
               "method": "pinned host x -> device -> moe_forward -> pinned host out, every step; steps pipelined "
                         "two deep on copy streams (events), one host wait after the last step; wall clock"}
        del x_host, out_host, x_dev, out_dev

    # ---- roofline of the dominant kernel (GEMM1: gate/up + SwiGLU; for
    # decode batches the fused expert FFN) ----
    kname = "ffn" if "ffn" in main_res["roofline"] else "gemm1"
    g1 = main_res["roofline"][kname]
    tkey = traffic_key(kname, w, main_res["tile_rows"])
    traffic, traffic_note = None, None
    if os.path.exists(TRAFFIC_FILE):
        tr = json.load(open(TRAFFIC_FILE))
        ent = tr.get("ratios", {}).get(tkey)
        if ent and tr.get("source_sha") == kernel_source_sha():
            traffic = ent["ratio"] * g1["algorithmic_bytes"]
            traffic_note = (f"DRAM bytes of {tkey} measured by ncu on {ent['workload']} ({ent['ratio']:.4f} x its "
                            "algorithmic bytes), scaled to this launch's algorithmic bytes")
    tensor_bound = g1["bound"] == "tensor"
    hbm = {"achieved": g1["gbs"], "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": g1["hbm_frac"],
           "algorithmic_bytes": g1["algorithmic_bytes"], "peak_source": pk["source"]}
    tensor = {"achieved": g1["tflops"], "peak": tpeak[w["fmt"]], "unit": "TFLOP/s", "frac": g1["tensor_frac"],
              "flops": g1["flops"], "peak_source": tsrc,
              "peak_note": "sustained block-scaled MMA rate of this GPU (moe_bench_mma_peak, "
                           f"{(mma or {}).get(w['fmt'], {}).get('mma', 'nominal ratio')}); the GEMM runs inside a "
                           "long run of steps"}
    top = tensor if tensor_bound else hbm
    roofline = {"bound": "tensor" if tensor_bound else "hbm",
                "kernel": "ffn_decode_fused" if kname == "ffn" else "gemm1_gate_up_swiglu",
                "achieved": top["achieved"], "peak": top["peak"], "unit": top["unit"], "frac": top["frac"],
                "traffic": traffic, "traffic_note": traffic_note, "peak_source": top["peak_source"], "hbm": hbm,
                "tensor": tensor,
                "gemm2": main_res["roofline"].get("gemm2"), "layer": main_res["roofline"]["layer"],
                "machine_balance_flop_per_byte": main_res["roofline"]["machine_balance_flop_per_byte"]}
    layer = {"us_per_layer": ms_per_step * 1e3, "step_us": step_dist, "stage_ms": main_res["stage_ms"]}

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_tok = 8 if T <= 1000 else 2
        samp = OracleSample(w, n_tok)
        # the same sample repeated until about 10 s of CPU work have been timed
        runs, t0 = 0, time.perf_counter()
        while True:
            samp.run()
            runs += 1
            dt = time.perf_counter() - t0
            if dt >= 10.0:
                break
        cpu = {"value": samp.tokens_per_call() * runs / dt, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{n_tok} tokens of {args.workload} through the whole layer ({samp.pairs} expert pairs, "
                         f"{len(samp.cache)} experts decoded on the fly), {runs} runs in {dt:.2f} s"}

    # ---- the other configurations (rank 0 of a single-GPU run) ----
    per = None
    if world == 1 and not args.no_per_workload:
        del gw
        torch.cuda.empty_cache()
        per = {}
        for nm, n_steps in PER_WORKLOAD.items():
            if nm == args.workload:
                continue
            g2w, r = measure_workload(moe, torch, nm, n_steps, max(args.warmup, 5), args.launch, tpeak,
                                      pk["hbm_gbs"], gpu_index, n_prof=50, ffn_schedule=args.ffn_schedule,
                                      y_format=args.y_format)
            rl = r["roofline"]
            per[nm] = {"T": r["T"], "fmt": r["fmt"], "touched_experts": r["touched_experts"], "steps": n_steps,
                       "ffn_schedule": r["ffn_schedule"],
                       "us_per_layer": r["us_per_layer"], "tokens_per_s": r["tokens_per_s"],
                       "bound": rl["layer"]["bound"], "layer_frac": rl["layer"]["frac"],
                       "stage_ms": r["stage_ms"], "clocks": r["clocks"]}
            for kn in ("ffn", "gemm1", "gemm2", "layer"):
                if kn in rl:
                    per[nm][kn + "_frac"] = rl[kn]["frac"]
                    per[nm][kn] = {k_: rl[kn][k_] for k_ in ("bound", "hbm_frac", "tensor_frac")}
            del g2w
            torch.cuda.empty_cache()

    kv = None
    if world == 1 and not args.no_per_workload:
        kv = measure_kv_quant(moe, torch, pk["hbm_gbs"])

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": w["fmt"], "data": "synthetic",
                "config": {"workload": args.workload, "T": T, "H": w["H"], "E": w["E"], "k": k, "F": w["F"],
                           "fmt": w["fmt"], "touched_experts": main_res["touched_experts"],
                           "parallelism": f"replicas{world}", "launch": main_res["launch"],
                           "ffn_schedule": main_res["ffn_schedule"], "y_format": main_res["y_format"],
                           "tile_rows": main_res["tile_rows"],
                           "l2": "inputs larger than L2: the touched expert weights of one step "
                                 f"({gemm_bytes(w, main_res['touched_experts'])[0] / 1e9:.2f} GB read by GEMM1 "
                                 "alone) against a 129 MB L2; no flush"},
                "layer": layer, "roofline": roofline, "tensor_peaks": mma, "cpu_baseline": cpu, "e2e": e2e,
                "per_workload": per, "kv_cache_quant_mxfp8": kv, "clocks": main_res["clocks"],
                "gpu_launches": main_res["gpu_launches"]}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
