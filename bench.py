#!/usr/bin/env python3
"""Benchmark of the K3-shape MXFP4 Stable LatentMoE routed-expert layer.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all|decode|chunk|prefill]
                [--impl ours|reference]

One step = one k3moe_forward over one batch of synthetic tokens (router, top-k,
permutation, latent down, expert gate/up + SiTU-GLU, expert down, combine, RMSNorm,
latent up), inputs resident in HBM.  L2 is flushed (256 MiB write) before every timed
step, outside the timed events.  Prints one JSON line (rank 0).

The default (--workload all) times the three K3-shape workloads one after another:
decode (1 token; the line's `value`, µs/token), then the 32-token chunk and the
4096-token prefill (`chunk` and `prefill` objects of the same line, with their own
value, roofline, phases, end-to-end time and oracle baseline).

--impl reference times the fp64 oracle on the host cores (the only reference this
method has), on a bounded sample of the same workload.
Under torchrun (N > 1) every rank runs an independent replica of the workload
(the layer does not shard across GPUs in this library); value aggregates all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "K3-shape MXFP4 LatentMoE layer: decode µs/token (HBM GB/s), prefill tokens/s"
FLUSH_BYTES = 256 << 20
WORKLOADS = ("decode", "chunk", "prefill", "decode_top_p", "prefill_mxfp8", "shared_decode", "shared_prefill")
DEFAULT_WORKLOADS = WORKLOADS
TOP_P = 0.7  # the pages' opt-in K3_TOPP setting


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", choices=("all",) + WORKLOADS, default="all")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="target CPU work of the oracle baseline, per workload and thread count")
    ap.add_argument("--no-graph", action="store_true", help="launch the forward eagerly instead of replaying a graph")
    ap.add_argument("--n-experts", type=int, default=None,
                    help="profiling case: a smaller expert pool with the same per-expert shapes and top-k")
    ap.add_argument("--tokens", type=int, default=None,
                    help="profiling case: this many tokens instead of the workload's")
    ap.add_argument("--sweep", type=str, default=None, metavar="T1,T2,...",
                    help="crossover sweep: time the forward at these token counts on both expert paths "
                         "(weight-streaming GEMVs and tensor-core GEMMs) and print one JSON line per count")
    ap.add_argument("--tc-min-tokens", type=int, default=None,
                    help="token count from which the tensor-core path runs (library default if omitted)")
    ap.add_argument("--tc-split-max-tokens", type=int, default=None,
                    help="token count below which the exact tensor-core expert GEMMs take the two-term "
                         "MXFP8 split (from it on the bf16 weight decode; 0 = never; library default if "
                         "omitted)")
    ap.add_argument("--no-flush", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--oracle-sample", choices=WORKLOADS, default=None, help=argparse.SUPPRESS)
    a = ap.parse_args(argv)
    a.warmup = max(a.warmup, 3)
    return a


def workload_cfg(name):
    import dataclasses
    from datagen import configs as C
    if name == "decode_top_p":  # decode with the experts pruned to cumulative weight TOP_P
        return dataclasses.replace(C.DECODE, name="decode_top_p", top_p=TOP_P)
    if name == "prefill_mxfp8":  # prefill with the low-precision-activation variant
        return dataclasses.replace(C.PREFILL, name="prefill_mxfp8", act_mxfp8=1)
    if name == "shared_decode":  # the fused shared experts beside the routed block, one token
        return dataclasses.replace(C.DECODE, name="shared_decode")
    if name == "shared_prefill":
        return dataclasses.replace(C.PREFILL, name="shared_prefill")
    return {"decode": C.DECODE, "chunk": C.CHUNK, "prefill": C.PREFILL}[name]


def selected_cfgs(a):
    """(name, config) of every workload this run times; the first one is the line's headline."""
    import dataclasses
    names = DEFAULT_WORKLOADS if a.workload == "all" else (a.workload,)
    out = []
    for n in names:
        cfg = workload_cfg(n)
        if a.n_experts:
            cfg = dataclasses.replace(cfg, n_experts=a.n_experts, name=cfg.name)
        if a.tokens:
            cfg = cfg.with_tokens(a.tokens, x_seed=cfg.x_seed)
        out.append((n, cfg))
    return out


def kernels_per_step(cfg, tc: bool, split_max: int = 1 << 30) -> int:
    """Kernel launches of one forward (the memsets are not kernels): for one token the
    router GEMV, then the routing and the latent down projection in one kernel (6 in all);
    up to 64 tokens the routing
    runs as one fused kernel (6 in all); beyond, top-k, the permutation (four
    kernels past 2 x 2048 routed slots, else one) and the activation prep (the f16 copy
    of z for the weight-streaming kernels, or on the grouped-GEMM path the slot-order
    gather), around the two projections, the two expert kernels and the combine."""
    if not tc and cfg.T == 1 and cfg.n_experts <= 1024 and cfg.top_k + 8 <= 32:
        return 6  # one token: router GEMV, then routing and latent down in one launch
    if not tc and cfg.T <= 64:
        return 6
    perm = 4 if cfg.T * cfg.top_k > 2 * 2048 else 1
    return 7 + perm + (splitk_reductions(cfg) + split_form(cfg, split_max) if tc else 0)


def split_form(cfg, split_max: int) -> bool:
    """The exact tensor-core experts take the two-term MXFP8 split below split_max tokens
    (k3moe_tc_split_max_tokens; one more launch: h's terms between the two GEMMs)."""
    return (cfg.T < split_max and not cfg.act_mxfp8 and cfg.latent >= 512 and cfg.inter >= 512)


def splitk_reductions(cfg, sms: int = 152) -> int:
    """The tensor-core projections split K over up to 8 CTAs per output tile when the tiles
    (128 tokens x 256 columns) number at most half the SMs (up to 512 tokens), each split
    launch followed by its reduction: the router + latent-down launch (E + L columns, K = H)
    and the latent up (H columns, K = L)."""
    if cfg.T > 512:
        return 0
    m = -(-cfg.T // 128)
    n = 0
    for cols, K in ((-(-cfg.n_experts // 256) + -(-cfg.latent // 256), cfg.hidden), (-(-cfg.hidden // 256), cfg.latent)):
        kb = K // 64
        n += any(2 * m * cols <= sms and kb % ks == 0 and kb // ks >= 4 for ks in (8, 4, 2))
    return n


def uses_grouped_gemm(cfg, tc_min_tokens: int) -> bool:
    """The library runs the experts on the grouped tcgen05 GEMM from tc_min_tokens tokens
    on (k3moe_tc_min_tokens) when both contraction lengths are multiples of 256; smaller
    batches stream the weights through the MXFP4 GEMV kernels."""
    return cfg.T >= tc_min_tokens and cfg.latent % 256 == 0 and cfg.inter % 256 == 0


def describe(cfg) -> str:
    if is_shared(cfg):
        from datagen import configs as C
        return (f"{cfg.name}: the 2 fused shared experts beside the routed block (SiTU-GLU on the hidden width), "
                f"T={cfg.T}, H={cfg.hidden}, fused width {C.SHARED_INTER}, bf16 weights, accumulated into the "
                f"block output")
    tp = f", top-p {cfg.top_p} (K3_TOPP)" if 0.0 < cfg.top_p < 1.0 else ""
    return (f"{cfg.name}: K3-shape routed layer, T={cfg.T}, H={cfg.hidden}, L={cfg.latent}, E={cfg.n_experts}, "
            f"K={cfg.top_k}{tp}, I={cfg.inter}, MXFP4 experts (scale bytes {cfg.scale_lo}..{cfg.scale_hi}), "
            f"bf16 latent projections" + (", MXFP8 expert activations (lossy variant)" if cfg.act_mxfp8 else ""))


def is_prefill(cfg) -> bool:
    return cfg.name.startswith("prefill") or cfg.name == "shared_prefill"


def is_shared(cfg) -> bool:
    return cfg.name.startswith("shared_")


def unit_of(cfg):
    return ("tokens/s", True) if is_prefill(cfg) else ("µs/token", False)


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest replica's time (the job ends when its last rank does): an all-reduce
    MAX over the default process group (NCCL tensors on `device`, or CPU for gloo)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def metric_value(cfg, ms_per_step, world):
    """Whole-job value of N replicas that each process cfg.T tokens per step."""
    if is_prefill(cfg):
        return cfg.T * world / (ms_per_step / 1e3)
    return ms_per_step * 1e3 / (cfg.T * world)


# ------------------------------------------------------------------------------ byte/flop model
def expert_bytes(cfg):
    I, L = cfg.inter, cfg.latent
    mat = I * L // 2 + I * L // 32  # one MXFP4 [I, L] or [L, I] matrix: packed + scales
    return 2 * mat, mat  # gate+up, down


def algorithmic(cfg, n_unique):
    """Algorithmic bytes (HBM) and flops per phase for one step."""
    T, H, L, E, K, I = cfg.T, cfg.hidden, cfg.latent, cfg.n_experts, cfg.top_k, cfg.inter
    gu, dn = expert_bytes(cfg)
    if cfg.act_mxfp8:  # the slot-order MXFP8 activation rows: one code byte + 1/32 scale byte
        za, ha = T * K * L * 33 // 32, T * K * I * 33 // 32
    else:
        za, ha = T * L * 2, T * K * I * 2
    return {
        "proj": dict(bytes=(E * H + L * H) * 2 + T * H * 2 + T * (E * 4 + L * 2), flops=2 * T * H * (E + L)),
        "gateup": dict(bytes=n_unique * gu + za + ha, flops=2 * T * K * 2 * I * L),
        "down": dict(bytes=n_unique * dn + ha + T * K * L * 4, flops=2 * T * K * L * I),
        "up": dict(bytes=H * L * 2 + T * L * 2 + T * H * 4, flops=2 * T * H * L),
    }


def step_flops(cfg):
    """Algorithmic flops of one forward: router + latent down, experts, latent up."""
    T, H, L, E, K, I = cfg.T, cfg.hidden, cfg.latent, cfg.n_experts, cfg.top_k, cfg.inter
    return 2 * T * (E * H + 2 * L * H + K * (2 * I * L + L * I))


def step_bytes(cfg, n_unique):
    """Algorithmic HBM bytes of one forward: dense weights once, the selected experts once."""
    gu, dn = expert_bytes(cfg)
    T, H, L, E = cfg.T, cfg.hidden, cfg.latent, cfg.n_experts
    return (E * H + 2 * L * H) * 2 + n_unique * (gu + dn) + T * H * (2 + 4)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            d = json.load(fh)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def tensor_peak(peaks):
    """The tensor denominator: the measured bf16 burst rate (a step of a few milliseconds is
    not a seconds-long loop).  The fraction against the sustained rate (the part at its power
    limit, as the prefill step runs: SM clocks near 1.8 GHz against 2.07) is reported beside
    it."""
    return peaks["bf16_tflops"], "bf16 burst"


def csrc_hash() -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "mxfp4_routed_expert_latentmoe_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh")):
            h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def profiled(kernel_phase, workload):
    """Figures recorded by an ncu capture under profiles/ (key: value lines), if the kernel
    sources are unchanged since the capture; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel_phase}_{workload}.md")
    try:
        kv = {}
        for line in open(path):
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("source_sha256_16") != csrc_hash():
            return None
        return kv
    except Exception:
        return None


def profiled_traffic(kernel_phase, workload):
    kv = profiled(kernel_phase, workload)
    try:
        return int(kv["dram_bytes_per_launch"]) if kv else None
    except (KeyError, ValueError):
        return None


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


# ------------------------------------------------------------------------------ raw CUDA events
class RawEvents:
    """Timing events created through the CUDA driver API, so that the C library can
    record them on its stream (handles are plain CUevent / cudaEvent_t)."""

    def __init__(self, n):
        import ctypes
        self.cu = ctypes.CDLL("libcuda.so.1")
        self.handles = []
        for _ in range(n):
            h = ctypes.c_void_p()
            if self.cu.cuEventCreate(ctypes.byref(h), 0) != 0:
                raise RuntimeError("cuEventCreate failed")
            self.handles.append(h)

    def ms(self, i, j) -> float:
        import ctypes
        v = ctypes.c_float()
        if self.cu.cuEventElapsedTime(ctypes.byref(v), self.handles[i], self.handles[j]) != 0:
            raise RuntimeError("cuEventElapsedTime failed")
        return float(v.value)

    def __del__(self):
        for h in getattr(self, "handles", []):
            self.cu.cuEventDestroy_v2(h)


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "20", "-i", gpu_id], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, windows):
        """Clock summary over the samples inside the given (t0, t1) windows."""
        if not self.samples:
            return None
        win = [p for (t, p) in self.samples if any(t0 <= t <= t1 for (t0, t1) in windows)]
        if not win:  # timed regions shorter than the sampling period: nearest samples
            win = [min(self.samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))[1] for (t0, t1) in windows]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        pw = [num(p[3]) for p in win if num(p[3]) is not None]
        reasons = set()
        for p in win:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), p[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons), "samples": len(win)}


# ------------------------------------------------------------------------------ oracle timing
def oracle_sample(cfg, seconds_target: float, min_tokens=1, max_tokens=64):
    """Times the oracle (token at a time, bf16-rounding spec mode) on a bounded sample of
    tokens drawn from the workload's recipe.  Returns (value in the metric's unit,
    threads, sample description, elapsed)."""
    import numpy as np
    import oracle
    from datagen import configs as C

    d = oracle.dims(**cfg.dims)
    x_all = C.layer_x(cfg)
    if is_shared(cfg):
        SW = C.shared_weights(cfg)

        def run(rows):
            x = np.ascontiguousarray(x_all[rows])
            t0 = time.perf_counter()
            oracle.shared(d, x, SW["wgu"], SW["wdn"], True)
            return time.perf_counter() - t0
    else:
        W = C.layer_weights(cfg)

        def run(rows):
            x = np.ascontiguousarray(x_all[rows])
            ids, _, _, _ = oracle.route(d, x, W["wr"], W["bias"])
            ex = {int(e): C.expert_tensors(cfg, int(e)) for e in np.unique(ids) if e >= 0}
            t0 = time.perf_counter()
            oracle.forward(d, x, W["wr"], W["bias"], W["wd"], W["wu"], W["gamma"], ex, True, 0)
            return time.perf_counter() - t0

    T = x_all.shape[0]
    t1 = run([0])
    n = int(max(min_tokens, min(max_tokens, T, seconds_target / max(t1, 1e-3))))
    rows = list(range(n)) if n <= T else [i % T for i in range(n)]
    el = run(rows)
    val = (n / el) if is_prefill(cfg) else (el / n * 1e6)
    return val, oracle.threads_used(), f"the first {n} token(s) of the {cfg.name} workload, token at a time", el


def oracle_baseline(cfg, unit, seconds):
    """The oracle on all host cores (in this process) and on one core (a child process
    with OMP_NUM_THREADS=1), each on a bounded token sample."""
    v, cores, sample, el = oracle_sample(cfg, seconds)
    out = {"value": v, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample, "seconds": el,
           "cpu": cpu_model()}
    try:
        env = dict(os.environ, OMP_NUM_THREADS="1")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", cfg.name,
                            "--cpu-seconds", str(seconds)], capture_output=True, text=True, env=env,
                           timeout=20 * seconds + 120)
        one = json.loads(r.stdout.strip().splitlines()[-1])
        out["single_thread"] = {"value": one["value"], "unit": unit, "cores": one["cores"], "sample": one["sample"],
                                "seconds": one["seconds"]}
    except Exception as e:  # the all-core figure stands on its own
        out["single_thread"] = {"error": f"{type(e).__name__}: {e}"[:200]}
    return out


# ------------------------------------------------------------------------------ reference arm
def run_reference(a, cfg, rank, world):
    unit, hib = unit_of(cfg)
    if rank != 0:
        return
    import numpy as np
    import oracle
    from datagen import configs as C
    oracle.build()
    d = oracle.dims(**cfg.dims)
    W = C.layer_weights(cfg)
    x_all = C.layer_x(cfg)
    per_step = 1 if not is_prefill(cfg) else 2
    steps = []
    rows_cycle = list(range(x_all.shape[0]))
    prepared = []
    for s in range(a.warmup + a.steps):
        rows = [rows_cycle[(s * per_step + j) % len(rows_cycle)] for j in range(per_step)]
        x = np.ascontiguousarray(x_all[rows])
        ids, _, _, _ = oracle.route(d, x, W["wr"], W["bias"])
        prepared.append((x, {int(e): C.expert_tensors(cfg, int(e)) for e in np.unique(ids) if e >= 0}))
        if len(prepared) > 8:
            break
    for s in range(a.warmup + a.steps):
        x, ex = prepared[s % len(prepared)]
        t0 = time.perf_counter()
        oracle.forward(d, x, W["wr"], W["bias"], W["wd"], W["wu"], W["gamma"], ex, True, 0)
        el = time.perf_counter() - t0
        if s >= a.warmup:
            steps.append(el)
    ms = statistics.mean(steps) * 1e3
    val = (per_step / (ms / 1e3)) if is_prefill(cfg) else ms * 1e3 / per_step
    cores = oracle.threads_used()
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": unit, "n_gpus": a.gpus, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": hib, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(cfg), "sample_tokens_per_step": per_step},
            "cpu_baseline": {"value": val, "unit": unit, "cores": cores, "kind": "oracle", "cpu": cpu_model(),
                             "sample": f"{per_step} token(s) per step of the {cfg.name} workload"},
            "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ our arm
def measure(a, cfg, k3, dev, world, pools, sampler):
    """Times one workload: the forward replayed from a CUDA graph (the figure), the same
    forward with per-phase events, and the end-to-end call with host buffers."""
    import numpy as np
    import torch
    import torch.distributed as dist
    from datagen import device as D

    unit, hib = unit_of(cfg)
    d = k3.dims(**cfg.dims)
    t = D.layer_tensors(cfg, dev)
    key = (cfg.seed, cfg.scale_lo, cfg.scale_hi, cfg.n_experts, cfg.latent, cfg.inter)
    if key not in pools:
        pools[key] = D.expert_pool(cfg, dev)
    pool, eb, offs = pools[key]
    tables = k3.ExpertTables.from_pool(pool, eb, offs)
    T = cfg.T
    out = torch.empty(T, cfg.hidden, dtype=torch.float32, device=dev)
    ids = torch.empty(T, cfg.top_k, dtype=torch.int32, device=dev)
    wts = torch.empty(T, cfg.top_k, dtype=torch.float32, device=dev)
    ws = torch.empty(k3.workspace_bytes(d, T), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    args = (d, t["x"], t["wr"], t["bias"], t["wd"], t["wu"], t["gamma"], tables, out, ws)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(a.warmup):
        flush.zero_()
        k3.forward(*args, ids_out=ids, w_out=wts)
    torch.cuda.synchronize()
    status = k3.device_status(ws)
    ids_h = ids.cpu().numpy()
    n_unique = int(np.unique(ids_h[ids_h >= 0]).size)

    # the timed step: one k3moe_forward captured into a CUDA graph (its kernels and
    # memsets, chained with programmatic dependent launch) and replayed
    step = lambda: k3.forward(*args, ids_out=ids, w_out=wts)
    graph = None
    if not a.no_graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream(dev).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        step = graph.replay
        for _ in range(a.warmup):
            flush.zero_()
            step()
        torch.cuda.synchronize()
    time.sleep(0.05)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    barrier()
    torch.cuda.synchronize()
    w0 = time.time()
    for s in range(a.steps):
        if not a.no_flush:
            flush.zero_()
        ev[s][0].record()
        step()
        ev[s][1].record()
    torch.cuda.synchronize()
    barrier()
    w1 = time.time()
    ms = max_over_ranks(statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev), world, dev)
    # per-kernel durations: events recorded by the library between phases, on its stream
    nph = len(k3.PHASES)
    pev = [RawEvents(nph + 1) for _ in range(a.steps)]
    torch.cuda.synchronize()
    for s in range(a.steps):
        if not a.no_flush:
            flush.zero_()
        k3.forward_profiled(*args, pev[s].handles, ids_out=ids, w_out=wts)
    torch.cuda.synchronize()
    phase_ms = {name: statistics.mean(pev[s].ms(i, i + 1) for s in range(a.steps)) for i, name in enumerate(k3.PHASES)}
    profiled_ms = statistics.mean(pev[s].ms(0, nph) for s in range(a.steps))

    # end to end through the public API with host buffers: H2D of x, the forward, D2H of out
    e2e = None
    if not a.no_e2e:
        xh = t["x"].cpu().pin_memory()
        oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        xd = torch.empty_like(t["x"])
        e2e_args = (d, xd) + args[2:]
        ms_e2e = []
        for s in range(a.warmup + max(10, a.steps // 4)):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            xd.copy_(xh, non_blocking=True)
            k3.forward(*e2e_args)
            oh.copy_(out, non_blocking=True)
            e1.record()
            e1.synchronize()
            if s >= a.warmup:
                ms_e2e.append(e0.elapsed_time(e1))
        me = max_over_ranks(statistics.mean(ms_e2e), world, dev)
        e2e = {"value": metric_value(cfg, me, world), "unit": unit, "h2d_bytes_per_step": xh.numel() * 2,
               "d2h_bytes_per_step": oh.numel() * 4, "ms_per_step": me}
    del ws, flush
    torch.cuda.empty_cache()

    peaks, peak_kind = measured_peaks()
    alg = algorithmic(cfg, n_unique)
    dom = "gateup"
    tc = uses_grouped_gemm(cfg, k3.tc_min_tokens())
    tpeak, tkind = tensor_peak(peaks)
    if tc and cfg.act_mxfp8:
        # block-scaled MMAs at the fp8 rate: peak = the measured bf16 rate x the nominal
        # 2x fp8/bf16 ratio; the weights also stream from HBM once -- report the tighter bound
        t_s = phase_ms[dom] / 1e3
        tf = alg[dom]["flops"] / t_s / 1e12
        gb = alg[dom]["bytes"] / t_s / 1e9
        fp8_peak = 2 * tpeak
        f_t, f_h = tf / fp8_peak, gb / peaks["hbm_gbs"]
        if f_h >= f_t:
            roof = {"bound": "hbm", "achieved": gb, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": f_h,
                    "peak_kind": f"{peak_kind} HBM copy"}
        else:
            roof = {"bound": "tensor", "achieved": tf, "peak": fp8_peak, "unit": "TFLOP/s", "frac": f_t,
                    "peak_kind": f"{peak_kind} {tkind} x 2 (nominal fp8/bf16 ratio)"}
        roof.update({"traffic": profiled_traffic(dom, cfg.name), "kernel": "k3_mx8_moe_kernel<0, 0> (gate/up)",
                     "other_bound_frac": f_t if f_h >= f_t else f_h,
                     "tflops_bf16_equivalent_frac": tf / tpeak})
    elif tc:
        # the grouped GEMM runs for milliseconds inside a step of a few milliseconds: the
        # burst bf16 rate is its tensor denominator (the sustained fraction is reported
        # beside it); with few tokens per expert (chunks) the weight bytes bound it instead
        # -- the tighter of the two is reported.  The split form does the bf16 products
        # exactly as two fp8 passes (twice the fp8 work at twice the bf16 rate): the
        # algorithmic flops against the bf16 rate are its bound too
        t_s = phase_ms[dom] / 1e3
        tf, gb = alg[dom]["flops"] / t_s / 1e12, alg[dom]["bytes"] / t_s / 1e9
        f_t, f_h = tf / tpeak, gb / peaks["hbm_gbs"]
        kv = profiled(dom, cfg.name) or {}
        if f_t >= f_h:
            roof = {"bound": "tensor", "achieved": tf, "peak": tpeak, "unit": "TFLOP/s", "frac": f_t,
                    "peak_kind": f"{peak_kind} {tkind}", "other_bound_frac": f_h,
                    "frac_vs_bf16_sustained": tf / peaks.get("bf16_tflops_sustained", tpeak)}
        else:
            roof = {"bound": "hbm", "achieved": gb, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": f_h,
                    "peak_kind": f"{peak_kind} HBM copy", "other_bound_frac": f_t}
        split = split_form(cfg, k3.tc_split_max_tokens())
        roof.update({"traffic": profiled_traffic(dom, cfg.name),
                     "kernel": "k3_mx8_moe_kernel<0, 1> (gate/up, exact two-term split)" if split
                     else "k3_tc_moe_kernel<0> (gate/up, bf16 weight decode)",
                     "tensor_pipe_active_pct": float(kv["tensor_pipe_active_pct"]) if "tensor_pipe_active_pct" in kv
                     else None})
    else:
        achieved = alg[dom]["bytes"] / (phase_ms[dom] / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": profiled_traffic(dom, cfg.name), "kernel": "k3_mxb_gemv_kernel<gate/up>",
                "peak_kind": f"{peak_kind} HBM copy"}
    phases = {k: {"us": v * 1e3,
                  "GB_s": (alg[k]["bytes"] / (v / 1e3) / 1e9) if k in alg else None,
                  "TFLOP_s": (alg[k]["flops"] / (v / 1e3) / 1e12) if k in alg else None}
              for k, v in phase_ms.items()}
    expert_us = (phase_ms["gateup"] + phase_ms["down"]) * 1e3
    exp_bytes = alg["gateup"]["bytes"] + alg["down"]["bytes"]
    res = {"value": metric_value(cfg, ms, world), "unit": unit, "higher_is_better": hib, "ms_per_step": ms,
           "config": {"workload": describe(cfg), "global_batch": cfg.T * world, "seq_len": cfg.T,
                      "parallelism": f"replicas x{world}", "l2": "flushed by a 256 MiB write before every timed step",
                      "unique_experts": n_unique, "experts_per_token": float((ids_h >= 0).sum()) / cfg.T,
                      "cuda_graph": graph is not None},
           "roofline": roof,
           "layer": {"GB_s": step_bytes(cfg, n_unique) / (ms / 1e3) / 1e9,
                     "frac_hbm": step_bytes(cfg, n_unique) / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                     "TFLOP_s": step_flops(cfg) / (ms / 1e3) / 1e12,
                     "frac_bf16_burst": step_flops(cfg) / (ms / 1e3) / 1e12 / peaks["bf16_tflops"],
                     "frac_bf16_sustained": step_flops(cfg) / (ms / 1e3) / 1e12 /
                                            peaks.get("bf16_tflops_sustained", tpeak)},
           "expert_phase": {"us": expert_us, "GB_s": exp_bytes / (expert_us / 1e6) / 1e9,
                            "frac_hbm": exp_bytes / (expert_us / 1e6) / 1e9 / peaks["hbm_gbs"]},
           "phases": phases, "profiled_ms_per_step": profiled_ms, "e2e": e2e,
           "gpu_launches": kernels_per_step(cfg, tc, k3.tc_split_max_tokens()) * a.steps, "device_status": status,
           "_window": (w0, w1)}
    return res


def sweep(a, local_rank):
    """The GEMV / tensor-core crossover: the whole forward of the prefill-shape layer at each
    token count, once with the tensor-core path forced off and forced on in each operand
    form of the exact grouped GEMM (the library's process-wide k3moe_set_tc_min_tokens and
    k3moe_set_tc_split_max_tokens), replayed from a CUDA graph with the L2 flushed before
    each step."""
    import torch

    import __graft_entry__ as g
    g.build()
    import mxfp4_routed_expert_latentmoe_gb300 as k3
    from datagen import configs as C
    from datagen import device as D

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    base = C.PREFILL
    pool, eb, offs = D.expert_pool(base, dev)
    tables = k3.ExpertTables.from_pool(pool, eb, offs)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    default, default_split = k3.tc_min_tokens(), k3.tc_split_max_tokens()
    for T in [int(v) for v in a.sweep.split(",")]:
        cfg = base.with_tokens(T, x_seed=base.x_seed)
        d = k3.dims(**cfg.dims)
        t = D.layer_tensors(cfg, dev)
        out = torch.empty(T, cfg.hidden, dtype=torch.float32, device=dev)
        row = {"sweep": "gemv_vs_tensor_core", "T": T, "default_tc_min_tokens": default}
        outs = {}
        for path, thr, split in (("gemv", 1 << 30, default_split), ("tc", 1, k3.SPLIT_ALWAYS), ("tc_decode", 1, 0)):
            k3.set_tc_min_tokens(thr)
            k3.set_tc_split_max_tokens(split)
            ws = torch.empty(k3.workspace_bytes(d, T), dtype=torch.uint8, device=dev)
            args = (d, t["x"], t["wr"], t["bias"], t["wd"], t["wu"], t["gamma"], tables, out, ws)
            for _ in range(a.warmup):
                k3.forward(*args)
            torch.cuda.synchronize()
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                k3.forward(*args)
            torch.cuda.current_stream(dev).wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                k3.forward(*args)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
            torch.cuda.synchronize()
            for s in range(a.steps):
                flush.zero_()
                ev[s][0].record()
                graph.replay()
                ev[s][1].record()
            torch.cuda.synchronize()
            ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
            row[f"{path}_us"] = ms * 1e3
            row[f"{path}_tokens_per_s"] = T / (ms / 1e3)
            row[f"{path}_device_status"] = k3.device_status(ws)
            outs[path] = out.clone()
            del graph, ws
        k3.set_tc_min_tokens(default)
        k3.set_tc_split_max_tokens(default_split)
        for path in ("tc", "tc_decode"):
            row[f"rel_l2_{path}_vs_gemv"] = ((outs[path] - outs["gemv"]).norm() / outs["gemv"].norm()).item()
        row["fastest"] = min(("gemv", "tc", "tc_decode"), key=lambda q: row[f"{q}_us"])
        print(json.dumps(row), flush=True)
        del t, out, outs
        torch.cuda.empty_cache()


def measure_shared(a, cfg, k3, dev, world):
    """Times k3moe_shared_forward (the fused shared experts accumulated into the output) on
    one workload: CUDA-graph replay with the L2 flushed, and end to end with host buffers."""
    import torch
    from datagen import configs as C
    from datagen import device as D

    unit, hib = unit_of(cfg)
    T, H, Is = cfg.T, cfg.hidden, C.SHARED_INTER
    d = k3.dims(**cfg.dims)
    SW = C.shared_weights(cfg, Is)
    wgu, wdn = D.bf16_tensor(SW["wgu"], dev), D.bf16_tensor(SW["wdn"], dev)
    x = D.bf16_tensor(C.layer_x(cfg), dev)
    out = torch.zeros(T, H, dtype=torch.float32, device=dev)
    ws = torch.empty(k3.shared_workspace_bytes(d, T, Is), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    step = lambda: k3.shared_forward(d, x, wgu, wdn, out, ws)
    for _ in range(a.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    status = k3.device_status(ws)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(a.warmup):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    w0 = time.time()
    for s in range(a.steps):
        flush.zero_()
        ev[s][0].record()
        graph.replay()
        ev[s][1].record()
    torch.cuda.synchronize()
    w1 = time.time()
    ms = max_over_ranks(statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev), world, dev)
    e2e = None
    if not a.no_e2e:
        xh = x.cpu().pin_memory()
        oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        xd = torch.empty_like(x)
        ms_e2e = []
        for s in range(a.warmup + max(10, a.steps // 4)):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            xd.copy_(xh, non_blocking=True)
            k3.shared_forward(d, xd, wgu, wdn, out, ws)
            oh.copy_(out, non_blocking=True)
            e1.record()
            e1.synchronize()
            if s >= a.warmup:
                ms_e2e.append(e0.elapsed_time(e1))
        me = max_over_ranks(statistics.mean(ms_e2e), world, dev)
        e2e = {"value": metric_value(cfg, me, world), "unit": unit, "h2d_bytes_per_step": xh.numel() * 2,
               "d2h_bytes_per_step": oh.numel() * 4, "ms_per_step": me}
    peaks, peak_kind = measured_peaks()
    wbytes = 3 * H * Is * 2
    bytes_ = wbytes + T * H * (2 + 4 + 4) + T * Is * (2 * 4 + 4 * 2 + 2 * 2)
    flops = 2 * T * 3 * H * Is
    gbs = bytes_ / (ms / 1e3) / 1e9
    tfs = flops / (ms / 1e3) / 1e12
    tpeak, tkind = tensor_peak(peaks)
    if T >= k3.tc_min_tokens():
        roof = {"bound": "tensor", "achieved": tfs, "peak": tpeak, "unit": "TFLOP/s",
                "frac": tfs / tpeak, "peak_kind": f"{peak_kind} {tkind}",
                "frac_vs_bf16_sustained": tfs / peaks.get("bf16_tflops_sustained", tpeak),
                "kernel": "whole call: k3_tc_dense_kernel<PLAIN>, k3_shared_glu_kernel, k3_tc_dense_kernel<ACC>"}
    else:
        roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "peak_kind": f"{peak_kind} HBM copy",
                "kernel": "whole call: dense GEMV<PLAIN>, k3_shared_glu_kernel, dense GEMV<ACC>"}
    roof["traffic"] = None
    roof["algorithmic_per_call"] = {"bytes": bytes_, "flops": flops}
    del ws, flush, wgu, wdn
    torch.cuda.empty_cache()
    return {"value": metric_value(cfg, ms, world), "unit": unit, "higher_is_better": hib, "ms_per_step": ms,
            "config": {"workload": describe(cfg), "global_batch": T * world, "seq_len": T,
                       "parallelism": f"replicas x{world}", "l2": "flushed by a 256 MiB write before every timed step",
                       "cuda_graph": True},
            "roofline": roof, "e2e": e2e, "gpu_launches": 3 * a.steps, "device_status": status,
            "_window": (w0, w1)}


def run_ours(a, cfgs, rank, world, local_rank):
    import torch

    import __graft_entry__ as g
    g.build()
    import mxfp4_routed_expert_latentmoe_gb300 as k3

    if a.tc_min_tokens:
        k3.set_tc_min_tokens(a.tc_min_tokens)
    if a.tc_split_max_tokens is not None:
        k3.set_tc_split_max_tokens(a.tc_split_max_tokens)
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(gpu_uuid if gpu_uuid.startswith("GPU-") else f"GPU-{gpu_uuid}")
    time.sleep(0.3)
    pools = {}
    results = {}
    for name, cfg in cfgs:
        results[name] = (measure_shared(a, cfg, k3, dev, world) if is_shared(cfg)
                         else measure(a, cfg, k3, dev, world, pools, sampler))
    time.sleep(0.1)
    sampler.stop()
    for r in results.values():
        r["clocks"] = sampler.summary([r.pop("_window")])
    per = [v["clocks"] for v in results.values()]
    if rank != 0:
        return
    if not a.no_cpu_baseline:
        for name, cfg in cfgs:
            results[name]["cpu_baseline"] = oracle_baseline(cfg, results[name]["unit"], a.cpu_seconds)
    head_name, head_cfg = cfgs[0]
    head = results[head_name]
    # the line's clocks: every timed region of the run
    reasons = sorted({x for c in per if c for x in c["reasons"]})
    sm = [c["sm_mhz"] for c in per if c and c["sm_mhz"] is not None]
    clocks = {"sm_mhz": statistics.median(sm) if sm else None,
              "sm_max_mhz": max((c["sm_max_mhz"] for c in per if c and c["sm_max_mhz"]), default=None),
              "reasons": reasons, "per_workload": {n: results[n]["clocks"] for n, _ in cfgs}}
    line = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": head["higher_is_better"],
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(head["config"], timed_workloads=[n for n, _ in cfgs]),
            "roofline": head["roofline"], "layer": head.get("layer"), "expert_phase": head.get("expert_phase"),
            "phases": head.get("phases"), "profiled_ms_per_step": head.get("profiled_ms_per_step"), "clocks": clocks,
            "e2e": head["e2e"], "gpu_launches": sum(results[n]["gpu_launches"] for n, _ in cfgs),
            "device_status": head["device_status"]}
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    for name, _cfg in cfgs[1:]:
        r = dict(results[name])
        line[name] = r
    print(json.dumps(line), flush=True)


def main():
    a = parse()
    if a.oracle_sample:  # child of oracle_baseline: one oracle sample, one JSON line
        cfg = workload_cfg(a.oracle_sample)
        v, cores, sample, el = oracle_sample(cfg, a.cpu_seconds)
        print(json.dumps({"value": v, "cores": cores, "sample": sample, "seconds": el}), flush=True)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if a.sweep:
        sweep(a, local_rank)
        return
    cfgs = selected_cfgs(a)
    if a.impl == "reference":
        run_reference(a, cfgs[0][1], rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(a, cfgs, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
