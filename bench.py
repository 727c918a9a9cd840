"""Benchmark of the KV-cache eviction pass on GB300.

Headline: the LORE-KV eviction pass (reliability weights, attention statistics, projected deletion
scores, chunked top-B selection and gather-compaction: lorekv_score + lorekv_select_compact) on
the Llama-3.1-8B-shaped 128K workload (1 sequence, 32 layers, 32/8 heads, d_head 128,
n = 131072, bf16). A step is one full pass over all 256 (layer, KV head) units; the metric is KV
tokens scored and compacted per second (a KV token = one (sequence, layer, KV head, position)).

Also reported: the H2O decode mode (OPT-30B shape: batch 64, 48 layers, 56 heads, d_head 128,
prompt 512, 512 decode steps) as KV tokens attended per second, and the fp64 oracle timed on the
host cores (cpu_baseline).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--no-h2o]
Under torchrun each rank runs its own sequence (the units are independent; no data exchange).
"""
from __future__ import annotations

import argparse
import csv
import dataclasses
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV tokens scored+compacted/sec (eviction pass, 128K ctx); % of HBM roofline"
UNIT = "tokens/s"
WORKLOAD = "llama"        # the 128K-context configuration the metric is quoted on

# DRAM bytes per launch of the dominant kernel from an ncu capture (--metrics
# dram__bytes_read.sum,dram__bytes_write.sum, one pass, full size), by (kernel, workload), with
# the hash of the kernel source file's code at capture time (src_hash: comments and whitespace
# left out); changed code reports null until re-captured. scores_tc_kernel: 128K workload
# 17.244 GB read + 0.535 GB written (K and V are 17.18 GB); Mistral-16K 2.207 + 0.065 GB
# (K + V 2.15 GB); Qwen 4 x 32K 26.492 + 1.004 GB (K + V 25.77 GB).
NCU_TRAFFIC = {("scores", "llama"): (17244091904 + 534949632, "a9ef66bf1aca8d1f"),
               ("scores", "mistral"): (2207387904 + 64717568, "a9ef66bf1aca8d1f"),
               ("scores", "qwen"): (26491987456 + 1004316416, "a9ef66bf1aca8d1f")}
# h2o_step_kernel on the OPT-30B shape at batch 8 (ncu, decode steps 21-23 after the 512-token
# prompt): 1.2094 GB read + 0.0268 GB written per launch against 1.2189 GB of algorithmic bytes
# (retained K/V rows, accumulated scores and positions, q/k/v/out): DRAM traffic is 1.014 x the
# algorithmic bytes, a ratio that holds at any batch and length (every term grows with the units
# and the retained rows), applied to the batch-64 launches.
NCU_TRAFFIC_H2O = (1.0146, "46dd9151c168d74b")
# cc_attn_tc_kernel on the n = 4096 counter-causal workload (ncu --set full, one launch):
# 37.807 MB read + 0.233 MB written
NCU_TRAFFIC_CC = {("cc_attention", "qwen7b_4096"): (37.80736e6 + 0.23296e6, "84e8ed792716cff5")}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--no-h2o", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-fidelity", action="store_true")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the other configured workloads (Mistral-16K, Qwen 4x32K, tiny)")
    p.add_argument("--no-cc", action="store_true", help="skip the counter-causal refresh")
    p.add_argument("--only-cc", action="store_true",
                   help="run only the counter-causal refresh and print its JSON (profiling)")
    p.add_argument("--cc-configs", default="qwen7b_512,qwen7b_4096",
                   help="counter-causal workloads (comma-separated names)")
    p.add_argument("--workload", default=WORKLOAD)
    p.add_argument("--h2o-batch", type=int, default=64, help="H2O batch (64 = OPT-30B workload)")
    p.add_argument("--h2o-steps", type=int, default=512, help="H2O decode steps")
    return p.parse_args()


# ---------------------------------------------------------------------------------------------
# distributed plumbing (host-side timing aggregation only)
# ---------------------------------------------------------------------------------------------
def dist_init(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return rank, world, local, pg


def whole_job_value(tokens_per_rank: float, world: int, ms: float) -> float:
    """Weak scaling over independent replicas: every rank scores its own sequence, so the job
    processes tokens_per_rank x world tokens in the slowest rank's time (ms)."""
    return tokens_per_rank * world / (ms / 1e3)


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, value: float, device=None) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if device is not None and pg.get_backend() == "nccl" else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        try:
            with open(self.path) as f:
                for r in csv.reader(f):
                    if len(r) >= 9:
                        rows.append([x.strip() for x in r])
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------------------------
# byte / flop accounting (per KV token-unit; a unit = one (sequence, layer, KV head))
# ---------------------------------------------------------------------------------------------
def lorekv_algorithmic_bytes(cfg) -> int:
    """K+V read once + Q_W + Q_look + logits + sampled ids read + compacted K', V' and kept
    indices written (scores and other intermediates are not counted)."""
    es = 2 if cfg.dtype == "bf16" else 4
    kv = 2 * cfg.units * cfg.n * cfg.d * es
    q = cfg.S * cfg.L * cfg.Hq * (cfg.w + cfg.M * cfg.T) * cfg.d * es
    logits = cfg.S * cfg.M * cfg.T * cfg.vocab * 4 + cfg.S * cfg.M * cfg.T * 4
    cap = cfg.n if cfg.n - cfg.sink - cfg.w <= cfg.B else cfg.sink + cfg.B + cfg.w
    out = 2 * cfg.units * cap * cfg.d * es + cfg.units * cap * 4
    return kv + q + logits + out


def scores_algorithmic_flops_per_token_unit(cfg) -> int:
    """The scoring kernel's algorithmic work per (token, unit): the cross term v.u_q for every
    query (2 g Qh d) and the quadratic form ||L_h^T v||^2 per query head (g d (d+1))."""
    Qh = cfg.w + cfg.M * cfg.T
    return 2 * cfg.g * Qh * cfg.d + cfg.g * cfg.d * (cfg.d + 1)


def scores_implemented_flops_per_token_unit(cfg) -> int:
    """MMA work the tensor-core scoring kernel (d = 128) executes per (token, unit), two query
    heads per CTA (64-query rows each): S = K [Q_h0;Q_h1]^T (N = 128) over K = 128 plus a
    constant-adding K step of 16; X = V U^T (128 columns) over K = 128; Y = V L_h of both heads in
    16-column groups that each run only the K steps at or after their diagonal block (Y_a: 26 and
    Y_b: 10 group-steps of 32 columns x 16); the constant-adding step over X | Y_a (N = 256)."""
    pairs = (cfg.g + 1) // 2
    per_pair = 128 * (128 + 16) + 128 * 128 + 32 * 16 * 26 + 32 * 16 * 10 + 256 * 16
    return 2 * pairs * per_pair


def attention_algorithmic_flops_per_token_unit(cfg) -> int:
    """q.k and the a.v accumulation for every query: 4 g Qh d."""
    Qh = cfg.w + cfg.M * cfg.T
    return 4 * cfg.g * Qh * cfg.d


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# GB300 FP32 FMA peak from unit counts and the maximum SM clock: 152 SMs x 128 FP32 lanes x 2
# flop x 2.07 GHz.
FP32_ALU_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def src_hash(rel):
    """sha256 prefix of a source file's code: comments removed and whitespace collapsed, so an ncu
    figure stays tied to the code it was taken on and survives edits to comments only."""
    import re
    with open(os.path.join(ROOT, rel)) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = re.sub(r"\s+", " ", text).strip()
    return hashlib.sha256(text.encode()).hexdigest()[:16]


# ---------------------------------------------------------------------------------------------
# the oracle as the CPU baseline / reference arm
# ---------------------------------------------------------------------------------------------
def oracle_sample(cfg, n_units: int, seed_layer: int = 0):
    """Inputs of a bounded sample of the workload (whole units), generated on the host."""
    import numpy as np
    import torch
    import oracle
    from kv_cache_eviction_02_gb300 import synth
    per_layer = cfg.Hkv
    layers = list(range(seed_layer, seed_layer + max(1, math.ceil(n_units / per_layer))))
    sub = cfg.replace(L=len(layers))
    # the sample's layers are generated with the same seeds as the full workload's first layers
    inp = synth.lorekv_inputs(sub, "cpu")
    units = [(0, l, kh) for l in range(len(layers)) for kh in range(cfg.Hkv)][:n_units]
    g, d = cfg.g, cfg.d
    prep = []
    for (s, l, kh) in units:
        u = synth.unit_slice(sub, inp, s, l, kh)
        Lf = np.stack([oracle.gram_cholesky(u["W_O"], d, kh * g + j)[1] for j in range(g)])
        prep.append((u, Lf))
    K = np.stack([oracle._d(u["K"]) for u, _ in prep])
    V = np.stack([oracle._d(u["V"]) for u, _ in prep])
    QW = np.stack([oracle._d(u["Q_W"]) for u, _ in prep])
    QL = np.stack([oracle._d(u["Q_look"]) for u, _ in prep])
    Lf = np.stack([lf for _, lf in prep])
    logits = oracle._d(inp["logits"][0])
    sampled = inp["sampled"][0].numpy()
    qlook_all = oracle._d(inp["Q_look"][0])
    del inp
    torch.set_num_threads(max(1, torch.get_num_threads()))
    return {"K": K, "V": V, "QW": QW, "QL": QL, "Lf": Lf, "logits": logits, "sampled": sampled,
            "qlook": qlook_all, "units": len(units)}


def oracle_step(cfg, smp):
    """One bounded oracle pass: reliability, scores of the sampled units (OpenMP over units),
    chunked top-B selection and gather."""
    import numpy as np
    import oracle
    om = oracle.reliability(smp["logits"], smp["sampled"], smp["qlook"], cfg.M, cfg.T, cfg.beta,
                            cfg.gamma, cfg.lambda_D)["omega"]
    S = oracle.lorekv_units(smp["K"], smp["V"], smp["QW"], smp["QL"], smp["Lf"],
                            np.tile(om, (smp["units"], 1)), M=cfg.M, T=cfg.T, sink=cfg.sink,
                            lambda_L=cfg.lambda_L, eps=cfg.eps, window_causal=cfg.window_causal)
    for u in range(smp["units"]):
        kept = oracle.select(S[u], sink=cfg.sink, w=cfg.w, chunk=cfg.chunk, B=cfg.B)
        oracle.compact(smp["K"][u], kept)
        oracle.compact(smp["V"][u], kept)
    return S


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_baseline(cfg, steps=1, warmup=0, one_core=True, n_tokens=None):
    """The oracle on the host cores: as many units as OpenMP threads (all cores busy), and, with
    one_core, a single unit (the OpenMP loop then keeps one core busy). n_tokens < cfg.n samples
    units of n_tokens tokens (a unit's pass costs in proportion to its tokens)."""
    import oracle
    threads = oracle.threads()
    full_n = cfg.n
    if n_tokens is not None and n_tokens < cfg.n:
        cfg = cfg.replace(n=n_tokens)
    smp = oracle_sample(cfg, threads)
    for _ in range(warmup):
        oracle_step(cfg, smp)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(cfg, smp)
    dt = (time.perf_counter() - t0) / steps
    tokens = smp["units"] * cfg.n
    res = {"value": tokens / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
           "sample": (f"{smp['units']} whole units (layer, KV head) of the {cfg.name} workload, "
                      f"{cfg.n} tokens each" if cfg.n == full_n else
                      f"{smp['units']} units (layer, KV head) of the {cfg.name} workload's shape "
                      f"with {cfg.n} of its {full_n} tokens each (a unit's pass costs in "
                      "proportion to its tokens)") +
                     ", reliability + scores + top-B + gather, fp64, OpenMP over units",
           "seconds_per_step": dt, "cpu_model": cpu_model()}
    if one_core:
        del smp
        smp1 = oracle_sample(cfg, 1)
        t0 = time.perf_counter()
        oracle_step(cfg, smp1)
        res["one_core_value"] = cfg.n / (time.perf_counter() - t0)
    return res


def run_reference(args):
    rank, world, local, pg = dist_init(args)
    from kv_cache_eviction_02_gb300 import synth
    cfg = synth.LOREKV_CONFIGS[args.workload]
    if rank != 0:
        barrier(pg)
        return
    # each step is a bounded sample: the units' token count is sized from a short calibration
    # step so that warm-up and timed steps together take about 100 s of host time
    steps_total = max(1, args.steps + args.warmup)
    cal = cpu_baseline(cfg, steps=1, warmup=0, one_core=False, n_tokens=4096)
    per_token_s = cal["seconds_per_step"] / 4096
    n_s = int(min(cfg.n, max(4096, (100.0 / steps_total) / per_token_s)))
    if n_s < cfg.n:  # a sample shorter than the workload: whole 4096-token blocks
        n_s = n_s // 4096 * 4096
    cb = cpu_baseline(cfg, steps=args.steps, warmup=args.warmup, one_core=False, n_tokens=n_s)
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": cb["seconds_per_step"] * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{cfg.name}: 1 seq x {cfg.L} layers x {cfg.Hq}/{cfg.Hkv} "
                                   f"heads, d_head {cfg.d}, n {cfg.n}, {cfg.dtype} inputs",
                       "sample": cb["sample"]},
            "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample",
                                                "cpu_model")},
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    barrier(pg)


# ---------------------------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------------------------
def measure_pass(cfg, g, dev, stream, pg, world, steps, warmup, pk, sample_clocks=None):
    """Times `steps` eviction passes (lorekv_score + lorekv_select_compact) on inputs `g` already
    resident in HBM, after `warmup` untimed passes; returns the bench fields of that workload
    (value, ms per step, HBM roofline, dominant-kernel roofline, stage times) plus the objects
    the later measurements reuse."""
    import torch
    from kv_cache_eviction_02_gb300 import api

    pb = api.LorekvProblem.from_config(cfg)
    Lf = torch.empty(cfg.L, cfg.Hq, cfg.d, cfg.d, device=dev)
    G = torch.empty_like(Lf)
    api.lorekv_prepare_wo(pb, g["W_O"], Lf, G)
    # per-model preparation, timed separately (warm: the second call)
    pw0 = torch.cuda.Event(enable_timing=True)
    pw1 = torch.cuda.Event(enable_timing=True)
    pw0.record(stream)
    api.lorekv_prepare_wo(pb, g["W_O"], Lf, G)
    pw1.record(stream)
    torch.cuda.synchronize(dev)
    prepare_wo_ms = pw0.elapsed_time(pw1)
    run = api.LorekvPass(pb, dev)
    for _ in range(warmup):
        run.run(g, Lf, G)
    api.kve_check_device()
    torch.cuda.synchronize(dev)

    # ---- timed region ----
    api.kve_profile_enable(True)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize(dev)
    # an event between consecutive steps as well, for the per-step spread (the steps still run
    # back to back; the first and last events bracket the timed region)
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(max(0, steps - 1))]
    clk = sample_clocks if sample_clocks is not None else _NoClock()
    with clk:
        ev0.record(stream)
        for k in range(steps):
            run.run(g, Lf, G)
            if k + 1 < steps:
                step_ev[k].record(stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    marks = [ev0] + step_ev + [ev1]
    step_ms = [a.elapsed_time(b) for a, b in zip(marks[:-1], marks[1:])]
    barrier(pg)
    api.kve_profile_enable(False)
    prof = api.kve_profile_report()
    api.kve_check_device()
    ms = ev0.elapsed_time(ev1) / steps
    ms = max_over_ranks(pg, ms, dev)
    tokens_per_step = cfg.units * cfg.n
    value = whole_job_value(tokens_per_step, world, ms)
    alg_bytes = lorekv_algorithmic_bytes(cfg)
    gpu_launches = sum(v["kernels"] for v in prof.values())

    # dominant kernel roofline (live CUDA-event timing of the kernel's launches)
    dom = max(prof, key=lambda k: prof[k]["ms"])
    dom_ms = prof[dom]["ms"] / prof[dom]["groups"]
    if dom == "scores":
        flops = scores_algorithmic_flops_per_token_unit(cfg) * tokens_per_step
    elif dom == "attention":
        flops = attention_algorithmic_flops_per_token_unit(cfg) * tokens_per_step
    else:
        flops = None
    tensor = cfg.dtype == "bf16" and cfg.d == 128 and cfg.w + cfg.M * cfg.T <= 64
    src = ("kv_cache_eviction_02_gb300/csrc/pass_tc.cu" if tensor
           else "kv_cache_eviction_02_gb300/csrc/pass_simt.cu")
    traffic = None
    key = (dom, cfg.name)
    if key in NCU_TRAFFIC and NCU_TRAFFIC[key][1] == src_hash(src):
        traffic = NCU_TRAFFIC[key][0]
    if flops is not None and tensor:
        # a step timed for well under a second: the burst bf16 figure applies
        ach = flops / (dom_ms / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops"], "traffic": traffic,
                "peak_source": f"bf16 dense burst, {pk['source']}", "ms_per_launch": dom_ms,
                "flops": "algorithmic"}
        if dom == "scores":  # what the kernel's MMAs execute (recomputed q.k, V L, constants)
            impl = scores_implemented_flops_per_token_unit(cfg) * tokens_per_step
            roof["implemented"] = {"flops": impl,
                                   "achieved": impl / (dom_ms / 1e3) / 1e12,
                                   "frac": impl / (dom_ms / 1e3) / 1e12 / pk["bf16_tflops"]}
    elif flops is not None:
        ach = flops / (dom_ms / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "alu", "achieved": ach, "peak": FP32_ALU_PEAK_TFLOPS,
                "unit": "TFLOP/s", "frac": ach / FP32_ALU_PEAK_TFLOPS, "traffic": traffic,
                "peak_source": "FP32 FMA: 152 SMs x 128 lanes x 2 flop x 2.07 GHz",
                "ms_per_launch": dom_ms}
    else:
        ach = alg_bytes / (dom_ms / 1e3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": ach / pk["hbm_gbs"], "traffic": traffic,
                "ms_per_launch": dom_ms}
    hbm_achieved = alg_bytes / (ms / 1e3) / 1e9
    pass_mma_flops = ((attention_algorithmic_flops_per_token_unit(cfg)
                       + scores_implemented_flops_per_token_unit(cfg)) * tokens_per_step)
    stages = {k: {"ms_per_step": v["ms"] / steps, "kernels": v["kernels"]}
              for k, v in prof.items()}
    out = {"value": value, "unit": UNIT, "ms_per_step": ms, "steps": steps, "warmup": warmup,
           "dtype": cfg.dtype,
           "workload": f"{cfg.name}: {cfg.S} seq x {cfg.L} layers x {cfg.Hq}/{cfg.Hkv} "
                       f"heads, d_head {cfg.d}, d_model {cfg.d_model}, n {cfg.n}, "
                       f"vocab {cfg.vocab}, w {cfg.w}, M {cfg.M}, T {cfg.T}, "
                       f"B {cfg.B}, chunk {cfg.chunk}, sink {cfg.sink}",
           "units": cfg.units, "kv_tokens_per_step": tokens_per_step,
           "hbm_roofline": {"algorithmic_bytes": alg_bytes, "achieved_gbs": hbm_achieved,
                            "peak_gbs": pk["hbm_gbs"], "frac": hbm_achieved / pk["hbm_gbs"],
                            "peak_source": pk["source"],
                            # the pass is a dense contraction: at the bf16 burst its MMA work
                            # alone takes t_min, which caps the HBM fraction
                            "ceiling_frac": (alg_bytes / (pass_mma_flops / (pk["bf16_tflops"] * 1e12))
                                             / 1e9 / pk["hbm_gbs"]) if tensor else None,
                            "pass_mma_flops": pass_mma_flops if tensor else None},
           "prepare_wo_ms": prepare_wo_ms,
           "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms),
                       "max": max(step_ms)},
           "roofline": roof, "stages": stages, "gpu_launches": gpu_launches}
    return out, run, Lf, G


class _NoClock:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


# the other configured workloads, reported beside the headline (name: timed steps)
OTHER_WORKLOADS = {"mistral": 20, "qwen": 6, "tiny": 50}


def run_native(args):
    import torch
    from kv_cache_eviction_02_gb300 import api, synth

    rank, world, local, pg = dist_init(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = synth.LOREKV_CONFIGS[args.workload]
    if world > 1:
        cfg = cfg.replace(seed=cfg.seed + rank)   # each rank scores its own sequence
    pk = peaks()
    stream = torch.cuda.current_stream(dev)

    # ---- inputs resident in HBM (17 GB per pass for the 128K workload: larger than L2) ----
    g = synth.lorekv_inputs(cfg, dev)
    clk = ClockSampler(local)   # nvidia-smi sampling during the timed passes only
    m, run, Lf, G = measure_pass(cfg, g, dev, stream, pg, world, args.steps, args.warmup, pk,
                                 sample_clocks=clk)
    alg_bytes = m["hbm_roofline"]["algorithmic_bytes"]
    line = {"metric": METRIC, "value": m["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.dtype, "data": "synthetic",
            "config": {"workload": m["workload"],
                       "units_per_gpu": cfg.units, "kv_tokens_per_step_per_gpu": m["kv_tokens_per_step"],
                       "l2": f"inputs larger than L2 ({alg_bytes / 1e9:.1f} GB per pass)",
                       "parallelism": f"replicas: {world} x independent sequence"},
            "hbm_roofline": m["hbm_roofline"], "prepare_wo_ms": m["prepare_wo_ms"],
            "step_ms": m["step_ms"], "roofline": m["roofline"], "stages": m["stages"],
            "gpu_launches": m["gpu_launches"], "clocks": clk.summary()}

    # ---- end to end through the public API with host buffers ----
    if not args.no_e2e:
        line["e2e"] = e2e_lorekv(cfg, g, run, Lf, G, dev, stream, pg, world, args)
    if not args.no_fidelity:
        line["fidelity"] = fidelity_lorekv(cfg, g, run, dev, stream)
    del g
    torch.cuda.empty_cache()

    if not args.no_workloads:
        line["workloads"] = {}
        for name, steps in OTHER_WORKLOADS.items():
            if name == cfg.name:
                continue
            wc = synth.LOREKV_CONFIGS[name]
            if world > 1:
                wc = wc.replace(seed=wc.seed + rank)
            wg = synth.lorekv_inputs(wc, dev)
            wm, wrun, _, _ = measure_pass(wc, wg, dev, stream, pg, world, steps,
                                          max(3, args.warmup), pk)
            line["workloads"][name] = wm
            del wg, wrun
            torch.cuda.empty_cache()
    if not args.no_h2o:
        line["h2o"] = bench_h2o(dev, stream, pg, world, args, pk)
    if not args.no_cc:
        line["cc_refresh"] = bench_cc(dev, stream, pg, args, pk)
        line["cc_cycle"] = bench_cc_cycle(dev, stream, pg, args)
    if rank == 0 and not args.no_cpu:
        try:
            cb = cpu_baseline(cfg)
            line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind",
                                                       "sample", "cpu_model", "one_core_value")}
        except Exception as e:  # the baseline is reported, never required
            line["cpu_baseline"] = {"value": None, "error": repr(e)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(pg)


def gpu_local_cpus(dev):
    """The host CPUs attached to the GPU's side of the machine (sysfs local_cpulist of its PCI
    function), limited to this process's allowed CPUs; None when unknown."""
    import torch
    p = torch.cuda.get_device_properties(dev)
    bus = getattr(p, "pci_bus_id", None)
    if bus is None:
        return None
    path = (f"/sys/bus/pci/devices/{getattr(p, 'pci_domain_id', 0):04x}:{bus:02x}:"
            f"{getattr(p, 'pci_device_id', 0):02x}.0/local_cpulist")
    try:
        with open(path) as f:
            text = f.read().strip()
    except OSError:
        return None
    cpus = set()
    for part in text.split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    cpus &= os.sched_getaffinity(0)
    return cpus or None


def _cpulist(text: str) -> set:
    cpus = set()
    for part in text.strip().split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    return cpus


def numa_report(dev) -> dict:
    """Where host memory and CPUs sit relative to the GPU: the GPU's NUMA node (sysfs of its PCI
    function) and, per node, the CPUs this process may use and the node's memory."""
    import torch
    out = {"gpu_node": None, "nodes": {}}
    p = torch.cuda.get_device_properties(dev)
    bus = getattr(p, "pci_bus_id", None)
    if bus is not None:
        path = (f"/sys/bus/pci/devices/{getattr(p, 'pci_domain_id', 0):04x}:{bus:02x}:"
                f"{getattr(p, 'pci_device_id', 0):02x}.0/numa_node")
        try:
            with open(path) as f:
                out["gpu_node"] = int(f.read().strip())
        except (OSError, ValueError):
            pass
    allowed = os.sched_getaffinity(0)
    base = "/sys/devices/system/node"
    try:
        names = sorted(x for x in os.listdir(base) if x.startswith("node") and x[4:].isdigit())
    except OSError:
        names = []
    for name in names:
        info = {}
        try:
            with open(os.path.join(base, name, "cpulist")) as f:
                info["cpus"] = len(_cpulist(f.read()) & allowed)
            with open(os.path.join(base, name, "meminfo")) as f:
                for ln in f:
                    if "MemTotal" in ln:
                        info["mem_gb"] = round(int(ln.split()[-2]) / 2**20, 1)
        except (OSError, ValueError):
            pass
        out["nodes"][name[4:]] = info
    return out


def e2e_lorekv(cfg, g, run, Lf, G, dev, stream, pg, world, args):
    """Host buffers in, host buffers out: per step the inputs are copied from pinned host memory,
    the pass runs, and the compressed cache is read back.

    Units are independent and, with lambda_D = 0, so is omega from the layers' queries, so one
    sequence's pass can be issued per chunk of layers through the same public calls
    (lorekv_score + lorekv_select_compact on the chunk's sub-shape): the copy of chunk j + 1 then
    runs on a second stream while chunk j is scored. Otherwise the whole pass is one call."""
    import torch
    from kv_cache_eviction_02_gb300 import api
    names = ["K", "V", "Q_W", "Q_look", "logits", "sampled"]
    layered = ["K", "V", "Q_W", "Q_look"]  # [S=1][L][...]: a layer chunk is contiguous
    # the pinned buffers are placed on the host memory next to this GPU: the allocating thread
    # runs on the GPU's local CPUs (pages land on the node of the thread that allocates them)
    old_aff = os.sched_getaffinity(0)
    local = gpu_local_cpus(dev)
    if local:
        os.sched_setaffinity(0, local)
    host = {k: torch.empty(g[k].shape, dtype=g[k].dtype, pin_memory=True) for k in names}
    for k in names:
        host[k].copy_(g[k])
    outs = [run.kept_idx, run.kept_len, run.K_out, run.V_out, run.omega]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    steps = max(1, min(args.steps, 3))
    cl = 4
    chunked = cfg.S == 1 and cfg.lambda_D == 0 and cfg.L % cl == 0 and cfg.L > cl
    if chunked:
        pb = api.LorekvProblem.from_config(cfg)
        sub = dataclasses.replace(pb, n_layers=cl)
        upc = cl * cfg.Hkv  # units per chunk
        ws = torch.empty(api.lorekv_workspace_size(sub), dtype=torch.uint8, device=dev)
        dev_in = [{k: torch.empty((1, cl) + tuple(g[k].shape[2:]), dtype=g[k].dtype, device=dev)
                   for k in layered} for _ in range(2)]
        small = {k: torch.empty_like(g[k]) for k in ("logits", "sampled")}
        cs = torch.cuda.Stream(dev)
        start_ev = torch.cuda.Event()
        copied = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        nch = cfg.L // cl
        scores = run.scores  # every chunk writes its slice of the full-size outputs

        # per-chunk timing: copy start/end on the copy stream, pass start/end on the compute
        # stream (timing events; recorded only when `marks` is given)
        def one(marks=None):
            start_ev.record(stream)
            if marks is not None:
                marks["t0"].record(stream)
            cs.wait_event(start_ev)
            # the logits and ids go first on the copy stream: the pass of chunk 0 waits on the
            # copy stream's event, which covers them (a copy queued on the compute stream behind
            # the copy engine's chunk copies would hold chunk 0's pass until the next chunk's copy)
            with torch.cuda.stream(cs):
                for k in ("logits", "sampled"):
                    small[k].copy_(host[k], non_blocking=True)
            for c in range(nch):
                b = c % 2
                if c >= 2:
                    cs.wait_event(done[b])  # chunk c - 2 has finished with buffer b
                with torch.cuda.stream(cs):
                    if marks is not None:
                        marks["copy"][c][0].record(cs)
                    for k in layered:
                        dev_in[b][k].copy_(host[k][:, c * cl:(c + 1) * cl], non_blocking=True)
                    copied[b].record(cs)
                    if marks is not None:
                        marks["copy"][c][1].record(cs)
                stream.wait_event(copied[b])
                if marks is not None:
                    marks["pass"][c][0].record(stream)
                x = dev_in[b]
                u0, u1 = c * upc, (c + 1) * upc
                sl = slice(c * cl, (c + 1) * cl)
                api.lorekv_score(sub, x["K"], x["V"], x["Q_W"], x["Q_look"], Lf[sl], G[sl],
                                 small["logits"], small["sampled"], scores[u0:u1], run.omega,
                                 ws, stream.cuda_stream)
                api.lorekv_select_compact(sub, scores[u0:u1], x["K"], x["V"], run.kept_idx[u0:u1],
                                          run.kept_len[u0:u1], run.K_out[u0:u1],
                                          run.V_out[u0:u1], None, stream.cuda_stream)
                done[b].record(stream)
                if marks is not None:
                    marks["pass"][c][1].record(stream)
            with torch.cuda.stream(stream):  # the step's results, read back once
                for t, h in zip(outs, host_out):
                    h.copy_(t, non_blocking=True)
    else:
        dev_in = {k: torch.empty_like(g[k]) for k in names}

        def one():
            with torch.cuda.stream(stream):
                for k in names:
                    dev_in[k].copy_(host[k], non_blocking=True)
            run.run(dev_in, Lf, G, stream.cuda_stream)
            with torch.cuda.stream(stream):
                for t, h in zip(outs, host_out):
                    h.copy_(t, non_blocking=True)

    one()
    torch.cuda.synchronize(dev)
    # the link's own rate on this machine: pinned host -> device copies of one layer's K
    probe_src = host["K"][:, 0]
    probe_dst = torch.empty(probe_src.shape, dtype=probe_src.dtype, device=dev)
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        p0.record(stream)
        for _ in range(4):
            probe_dst.copy_(probe_src, non_blocking=True)
        p1.record(stream)
    torch.cuda.synchronize(dev)
    link_gbs = 4 * probe_src.numel() * probe_src.element_size() / (p0.elapsed_time(p1) / 1e3) / 1e9
    del probe_dst
    barrier(pg)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    se = [ev() for _ in range(steps + 1)]
    # every timed step carries its per-chunk marks (copy start/end on the copy stream, pass
    # start/end on the compute stream): a slow step shows which copies were slow
    marks = [{"t0": ev(), "copy": [(ev(), ev()) for _ in range(nch)],
              "pass": [(ev(), ev()) for _ in range(nch)]} if chunked else None
             for _ in range(steps)]
    se[0].record(stream)
    for i in range(steps):
        if chunked:
            one(marks[i])
        else:
            one()
        se[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(pg, se[0].elapsed_time(se[steps]) / steps, dev)
    step_ms = [round(se[i].elapsed_time(se[i + 1]), 3) for i in range(steps)]
    timeline = None
    if chunked:
        chunk_bytes = sum(host[k][:, :cl].numel() * host[k].element_size() for k in layered)

        def rates(mk):
            return [round(chunk_bytes / (a.elapsed_time(b) / 1e3) / 1e9, 1) for a, b in mk["copy"]]

        slow = max(range(steps), key=lambda i: step_ms[i])
        mk = marks[slow]
        t0 = mk["t0"]
        timeline = {
            "chunk_bytes": chunk_bytes,
            "copy_gbs_by_step": [rates(m) for m in marks],
            "slowest_step": slow,
            "copy_ms": [[round(t0.elapsed_time(a), 3), round(t0.elapsed_time(b), 3)]
                        for a, b in mk["copy"]],
            "pass_ms": [[round(t0.elapsed_time(a), 3), round(t0.elapsed_time(b), 3)]
                        for a, b in mk["pass"]],
            "note": "copy_ms / pass_ms: the slowest timed step, ms from its start (copy: copy "
                    "stream, pass: compute stream); copy_gbs_by_step: each chunk's copy rate in "
                    "every timed step",
        }
    del host, dev_in
    os.sched_setaffinity(0, old_aff)
    res = {"value": cfg.units * cfg.n * world / (ms / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
           "steps": steps, "step_ms": step_ms, "h2d_gbs_effective": h2d / (ms / 1e3) / 1e9,
           "link_probe_gbs": link_gbs,
           "numa": numa_report(dev)}
    if chunked:
        res["issue"] = (f"{cfg.L // cl} chunks of {cl} layers: the next chunk's host-to-device "
                        "copy overlaps the current chunk's pass (copy stream + compute stream)")
        res["timeline"] = timeline
    res["host_buffers"] = (f"pinned, allocated from the GPU's local CPUs ({len(local)} CPUs)"
                           if local else "pinned (GPU-local CPUs unknown)")
    return res


def fidelity_lorekv(cfg, g, run, dev, stream):
    """Attention-output fidelity of the compressed cache (the diagnostic on top of the attention
    statistics): queries attend over the full K/V and over the compacted K'/V' (both seeing the
    whole cache), then the per-query cosine of the two outputs and its mean. Two query sets: the
    generator's queries under another seed (held out), and the window and lookahead queries the
    scores were computed from (in sample). Timed once, outside the pass's timed region."""
    import torch
    from kv_cache_eviction_02_gb300 import api, synth
    held = synth.lorekv_inputs(cfg.replace(seed=cfg.seed + 1000), dev)
    sets = {"held_out": (held["Q_W"], held["Q_look"]), "in_sample": (g["Q_W"], g["Q_look"])}
    del held
    torch.cuda.empty_cache()
    pe = dataclasses.replace(api.LorekvProblem.from_config(cfg), window_causal=0)
    pc = dataclasses.replace(pe, n_tokens=run.cap)
    qu = cfg.g * cfg.queries_per_head
    lse = torch.empty(cfg.units, qu, device=dev)
    o_full = torch.empty(cfg.units, qu, cfg.d, device=dev)
    o_comp = torch.empty_like(o_full)
    ws = torch.empty(api.lorekv_workspace_size(pe), dtype=torch.uint8, device=dev)
    wsc = torch.empty(api.lorekv_workspace_size(pc), dtype=torch.uint8, device=dev)
    cos = torch.empty(cfg.units * qu, device=dev)
    mean = torch.empty(1, device=dev)
    out = {"definition": "cosine between a query's attention output over the compacted cache "
                         f"({run.cap} tokens per unit) and over the full cache",
           "note": "the synthetic keys give no query a few dominant tokens (77 % of keys share "
                   "the largest Zipf bias), so attention spreads over ~1e5 tokens and a 164-token "
                   "cache cannot reproduce it; the LORE-KV page's 0.873 -> 0.905 (Attention-output "
                   "fidelity) are on LongBench text"}
    for name, (Qw, Ql) in sets.items():
        def one():
            api.lorekv_attention_stats(pe, g["K"], g["V"], Qw, Ql, lse, o_full, ws, stream)
            api.lorekv_attention_stats(pc, run.K_out, run.V_out, Qw, Ql, lse, o_comp, wsc,
                                       stream)
            api.lorekv_output_fidelity(o_full.view(-1, cfg.d), o_comp.view(-1, cfg.d), cos,
                                       mean, stream)
        one()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        one()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        api.kve_check_device()
        c = cos.float()
        out[name] = {"mean_cosine": float(mean.item()), "p05_cosine": float(torch.quantile(c, 0.05)),
                     "queries": int(c.numel()), "ms": e0.elapsed_time(e1)}
    return out


def bench_h2o(dev, stream, pg, world, args, pk):
    """H2O decode on the OPT-30B shape: prefill once (timed separately), then the decode steps
    with the first `warmup` steps untimed."""
    import torch
    from kv_cache_eviction_02_gb300 import api, synth
    cfg = synth.H2O_CONFIGS["opt30b"].replace(batch=args.h2o_batch, steps=args.h2o_steps)
    hin = synth.h2o_inputs(cfg, dev)
    # the state owns every buffer the prefill and the decode steps use (created, and touched,
    # before the timed region): the timed prefill allocates nothing
    st = api.h2o_state_create(cfg.batch, cfg.L, cfg.H, cfg.d, cfg.prompt + cfg.steps,
                              cfg.budget_frac, torch.float16)
    api.kve_profile_enable(True)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    st.prefill(hin["K"], hin["V"], hin["Q"])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    prefill_ms = e0.elapsed_time(e1)
    api.kve_profile_report()
    out = torch.empty(cfg.batch, cfg.L, cfg.H, cfg.d, dtype=torch.float16, device=dev)
    w = min(max(args.warmup, 3), cfg.steps - 1)
    for t in range(w):
        st.decode_step(hin["q"][t], hin["k"][t], hin["v"][t], out)
    torch.cuda.synchronize(dev)
    barrier(pg)
    e0.record(stream)
    for t in range(w, cfg.steps):
        st.decode_step(hin["q"][t], hin["k"][t], hin["v"][t], out)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    api.kve_profile_enable(False)
    prof = api.kve_profile_report()
    steps = cfg.steps - w
    ms = max_over_ranks(pg, e0.elapsed_time(e1) / steps, dev)
    # tokens attended per step: after appending at length t the unit holds floor(0.2 (t-1)) + 1
    held = [math.floor(cfg.budget_frac * (cfg.prompt + s)) + 1 for s in range(w, cfg.steps)]
    tokens = cfg.units * sum(held) / steps
    row = 2 * cfg.d * 2            # K and V row bytes
    per_step_bytes = cfg.units * (sum(held) / steps * (row + 8) + 4 * cfg.d * 2 + 16)
    step_ms = prof["h2o_step"]["ms"] / prof["h2o_step"]["groups"]
    ach = per_step_bytes / (step_ms / 1e3) / 1e9
    st.close()
    del hin
    torch.cuda.empty_cache()
    # prefill: bound by HBM. At d_head 128 the causal q.k is about 128 flop per byte of Q and K,
    # below the bf16 ridge (about 280 flop/B). Algorithmic bytes: Q and K read once, the kept
    # rows' K and V read and written once, the kept accumulated scores and positions written.
    # The tensor figures (one q.k over the causal triangle; the kernels' 128 x 128 x 128 blocks
    # over every (query tile, key tile <= it) pair) are reported beside it.
    nt = (cfg.prompt + 127) // 128
    keep = math.floor(cfg.budget_frac * cfg.prompt)
    es = 2
    pf_bytes = cfg.units * (2 * cfg.prompt * cfg.d * es + 4 * keep * cfg.d * es + 8 * keep)
    pf_impl = cfg.units * 2 * (nt * (nt + 1) // 2) * 2 * 128 ** 3
    pf_alg = cfg.units * (cfg.prompt * (cfg.prompt + 1) // 2) * 2 * cfg.d
    pf_s = prefill_ms / 1e3
    pf_roof = {"kernel": "h2o prefill (column sums + compression)", "bound": "hbm",
               "achieved": pf_bytes / pf_s / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
               "frac": pf_bytes / pf_s / 1e9 / pk["hbm_gbs"], "bytes": pf_bytes,
               "tensor_tflops_algorithmic": pf_alg / pf_s / 1e12,
               "tensor_frac_algorithmic": pf_alg / pf_s / 1e12 / pk["bf16_tflops"],
               "tensor_frac_implemented": pf_impl / pf_s / 1e12 / pk["bf16_tflops"]}
    return {"metric": "KV tokens attended+scored/sec (H2O decode step)",
            "value": tokens * world / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "steps": steps, "warmup": w, "prefill_ms": prefill_ms, "prefill_roofline": pf_roof,
            "config": f"{cfg.name}: batch {cfg.batch}, {cfg.L} layers, {cfg.H} heads, d_head {cfg.d}, "
                      f"prompt {cfg.prompt}, {cfg.steps} decode steps, budget 20%, fp16",
            "roofline": {"kernel": "h2o_step", "bound": "hbm", "achieved": ach,
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"],
                         "traffic": (NCU_TRAFFIC_H2O[0] * per_step_bytes
                                     if NCU_TRAFFIC_H2O[1] == src_hash("kv_cache_eviction_02_gb300/csrc/h2o.cu")
                                     else None),
                         "bytes_per_launch": per_step_bytes}}


# Counter-causal refresh latency of the fast single-layer variant on the page's own setup (Qwen2.5-
# 7B, fp16, RTX 4090; review of "Back from the Future", Table 1): context, not a target.
CC_PAGE_MS = {"qwen7b_512": 7.9, "qwen7b_4096": 52.6}


def cc_attention_flops(cfg) -> int:
    """Counter-causal attention: per query head and visible (i, j > i) pair, q.k and p v."""
    return cfg.batch * cfg.Hq * (cfg.n * (cfg.n - 1) // 2) * 4 * cfg.d


def cc_logits_flops(cfg) -> int:
    """r = h + W_O o over all tokens, then the true token's logit W_U[x] . r."""
    return cfg.batch * cfg.n * (2 * cfg.d_model * cfg.Hq * cfg.d + 2 * cfg.d_model)


def bench_cc(dev, stream, pg, args, pk):
    """Counter-causal surprise refresh (fast single-layer variant): cc_surprise +
    cc_select_compact on the Qwen2.5-7B-shaped last layer at n = 512 and 4096. Each refresh is
    timed alone with CUDA events after a 256 MB write that flushes L2 (the inputs fit in it)."""
    import torch
    from kv_cache_eviction_02_gb300 import api, synth
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    for name in args.cc_configs.split(","):
        cfg = synth.CC_CONFIGS[name]
        inp = synth.cc_inputs(cfg, dev)
        pb = api.CcProblem(cfg.batch, cfg.Hq, cfg.Hkv, cfg.d, cfg.d_model, cfg.n, cfg.vocab,
                           api.KVE_BF16, cfg.sink, cfg.J)
        ws = torch.empty(api.cc_workspace_size(pb), dtype=torch.uint8, device=dev)
        s = torch.empty(cfg.batch, cfg.n, dtype=torch.float32, device=dev)
        kept = torch.empty(cfg.batch, cfg.J, dtype=torch.int32, device=dev)
        Ko = torch.empty(cfg.batch, cfg.Hkv, cfg.J, cfg.d, dtype=torch.bfloat16, device=dev)
        Vo = torch.empty_like(Ko)
        Xo = torch.empty(cfg.batch, cfg.J, dtype=torch.int32, device=dev)

        def refresh():
            api.cc_surprise(pb, inp["K"], inp["V"], inp["Q_fresh"], inp["H_last"], inp["W_O"],
                            inp["W_U"], inp["tokens"], s, ws, stream)
            api.cc_select_compact(pb, s, inp["K"], inp["V"], inp["tokens"], kept, Ko, Vo, Xo,
                                  stream)

        for _ in range(max(args.warmup, 3)):
            refresh()
        api.kve_check_device()
        steps = max(1, min(args.steps, 20))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        barrier(pg)
        torch.cuda.synchronize(dev)
        api.kve_profile_enable(True)
        with ClockSampler(dev.index) as clk:
            for e0, e1 in ev:
                with torch.cuda.stream(stream):
                    flush.zero_()
                e0.record(stream)
                refresh()
                e1.record(stream)
            torch.cuda.synchronize(dev)
        api.kve_profile_enable(False)
        prof = api.kve_profile_report()
        api.kve_check_device()
        ms = max_over_ranks(pg, sum(a.elapsed_time(b) for a, b in ev) / steps, dev)
        stages = {k: v["ms"] / v["groups"] for k, v in prof.items()}
        ck = clk.summary()
        att_ms = stages.get("cc_attention")
        ach = cc_attention_flops(cfg) / (att_ms / 1e3) / 1e12 if att_ms else None
        # bf16 with d_head 128 runs on the tensor cores: a kernel timed alone, the burst peak
        traffic = None
        key = ("cc_attention", name)
        if key in NCU_TRAFFIC_CC and NCU_TRAFFIC_CC[key][1] == src_hash(
                "kv_cache_eviction_02_gb300/csrc/cc_tc.cu"):
            traffic = NCU_TRAFFIC_CC[key][0]
        att_roof = {"kernel": "cc_attention", "bound": "tensor", "achieved": ach,
                    "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": ach / pk["bf16_tflops"] if ach else None, "traffic": traffic,
                    "peak_source": f"bf16 dense burst, {pk['source']}",
                    "flops": cc_attention_flops(cfg), "ms_per_launch": att_ms}
        out[name] = {
            "ms_per_refresh": ms, "steps": steps,
            "config": f"{name}: batch {cfg.batch}, {cfg.Hq}/{cfg.Hkv} heads, d_head {cfg.d}, "
                      f"d_model {cfg.d_model}, vocab {cfg.vocab}, n {cfg.n}, keep J {cfg.J}, "
                      f"sink {cfg.sink}, bf16; L2 flushed before each refresh",
            "stages_ms": stages,
            "gpu_launches_per_refresh": sum(v["kernels"] for v in prof.values()) // steps,
            "page_ms_rtx4090_fp16": CC_PAGE_MS[name],
            "roofline": att_roof,
            "logits_tflops": (cc_logits_flops(cfg) / (stages["cc_logits"] / 1e3) / 1e12
                              if stages.get("cc_logits") else None),
            "clocks": ck}
        del inp, ws, s, kept, Ko, Vo, Xo
        torch.cuda.empty_cache()
    del flush
    torch.cuda.empty_cache()
    return out


def bench_cc_cycle(dev, stream, pg, args, J=512, h=128):
    """Counter-causal refresh cycle (Algorithms 1 and 3 without the model) on the
    Qwen2.5-7B-shaped last layer: memory J = 512, chunk h = J/4. Tokens of a seeded stream enter
    in appends of h; each timed iteration is one append of h tokens plus the refresh over the
    J + h candidates (with evictions), timed alone with CUDA events after a 256 MB L2 flush."""
    import torch
    from kv_cache_eviction_02_gb300 import api, synth
    warm = max(args.warmup, 3)
    steps = max(1, min(args.steps, 20))
    T = J + h * (warm + steps)
    cfg = synth.CC_CONFIGS["qwen7b_512"].replace(name="qwen7b_cycle", n=T, J=J)
    inp = synth.cc_inputs(cfg, dev)
    pb = api.CcProblem(cfg.batch, cfg.Hq, cfg.Hkv, cfg.d, cfg.d_model, J + h, cfg.vocab,
                       api.KVE_BF16, cfg.sink, J)
    cache = api.CcCache(pb)
    chunks = [[inp[k][:, :, i:i + h].contiguous() if k in ("K", "V", "Q_fresh")
               else inp[k][:, i:i + h].contiguous()
               for k in ("K", "V", "Q_fresh", "H_last", "tokens")] for i in range(0, T, h)]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    it = 0
    while it < J // h + warm:  # fill the memory (no evictions), then warm-up refreshes
        assert cache.step(*chunks[it], inp["W_O"], inp["W_U"], stream)
        it += 1
    api.kve_check_device()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier(pg)
    torch.cuda.synchronize(dev)
    api.kve_profile_enable(True)
    for e0, e1 in ev:
        with torch.cuda.stream(stream):
            flush.zero_()
        e0.record(stream)
        cache.step(*chunks[it], inp["W_O"], inp["W_U"], stream)
        e1.record(stream)
        it += 1
    torch.cuda.synchronize(dev)
    api.kve_profile_enable(False)
    prof = api.kve_profile_report()
    api.kve_check_device()
    ms = max_over_ranks(pg, sum(a.elapsed_time(b) for a, b in ev) / steps, dev)
    cache.close()
    del inp, chunks, flush
    torch.cuda.empty_cache()
    return {"ms_per_cycle": ms, "steps": steps, "tokens_per_s": h / (ms / 1e3),
            "stages_ms": {k: v["ms"] / v["groups"] for k, v in prof.items()},
            "gpu_launches_per_cycle": sum(v["kernels"] for v in prof.values()) // steps,
            "config": f"qwen7b cycle: batch 1, 28/4 heads, d_head 128, d_model 3584, vocab "
                      f"152064, memory J {J}, chunk h {h} (J + h = {J + h} candidates), sink 4, "
                      "bf16; one append of h tokens + one refresh per cycle; L2 flushed before "
                      "each cycle",
            "page_ms_rtx4090_fp16": {"refresh n=512": CC_PAGE_MS["qwen7b_512"]}}


def run_cc_only(args):
    import torch
    rank, world, local, pg = dist_init(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    st = torch.cuda.current_stream(dev)
    out = {"cc_refresh": bench_cc(dev, st, pg, args, peaks()),
           "cc_cycle": bench_cc_cycle(dev, st, pg, args)}
    if rank == 0:
        print(json.dumps(out), flush=True)
    barrier(pg)


def main():
    args = parse()
    if args.only_cc and args.impl != "reference":
        run_cc_only(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
