#!/usr/bin/env python
"""Benchmark: sparse MoE layer forward, tokens/s on B300, against its roofline.

Default workload: the Mixtral-shaped prefill layer (T=4096, d=4096, 8 experts,
SiLU-gated hidden 14336, top-2, top-k then softmax; bf16 activations and experts,
fp32 router). One step = one moe_forward over the whole batch: router, gating,
counts and aux loss, dispatch, both expert products on tensor cores, combine.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   (the CPU oracle, timed on host cores)

Multi-GPU (torchrun, one process per GPU): every rank runs an independent replica
of the layer on its own batch (the layer needs no exchange between replicas);
the time is the max over ranks and `value` counts the tokens of all ranks.

On one GPU the default run also measures the layer's other workloads (the
DeepSeekMoE-shaped layer, Mixtral-shaped decode at T = 16, 64 and 128, Switch
top-1 with capacity, tiny fp32, Expert Choice routing of the Mixtral-shaped layer)
the same way, each under "workloads" in the same line, with its own oracle baseline
on a bounded sample.

Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


# The CPU oracle's float64 numpy work runs on every core this process may use: the
# BLAS pool size is fixed when numpy's OpenBLAS loads, so it is set before the import.
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_host_cores()))

import torch  # noqa: E402

import workloads as W  # noqa: E402

L2_BYTES = 126 * 1024 * 1024
METRIC = "MoE layer tokens/s on 1 B300 and % of roofline (BF16 TC peak / HBM BW)"
UNIT = "tokens/s"
STAGES = ["router", "dispatch", "expert_product_1", "expert_product_2", "combine"]


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="mixtral_prefill", choices=sorted(W.WORKLOADS))
    ap.add_argument("--tokens", type=int, default=None, help="override T (profiling variants)")
    ap.add_argument("--experts", type=int, default=None, help="override N (profiling variants)")
    ap.add_argument("--hidden", type=int, default=None, help="override h (profiling variants)")
    ap.add_argument("--cpu-sample", type=int, default=1024,
                    help="tokens whose outputs the CPU oracle computes for cpu_baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="repeat oracle passes (new token samples) until this much CPU time is spent")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the training-router, sharded-router and backward variant timing")
    ap.add_argument("--workloads", default="auto", choices=["auto", "all", "none"],
                    help="also measure the other workloads of the layer (auto: when the default "
                         "workload runs on one GPU without overrides)")
    ap.add_argument("--secondary-cpu-seconds", type=float, default=2.0,
                    help="CPU seconds of the oracle baseline for each of the other workloads")
    return ap.parse_args()


# The other workloads measured in the same run as the default one (one GPU): every
# configuration the layer is specified on besides the Mixtral-shaped prefill layer, and
# Expert Choice routing of that layer.
SECONDARY = ["deepseek_fine", "mixtral_decode_16", "mixtral_decode_64", "mixtral_decode_128",
             "switch_top1", "tiny_fp32", "mixtral_expert_choice"]


# --------------------------------------------------------------------------- helpers

def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)
    return world, rank, local


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def _max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    dev = "cuda" if torch.cuda.is_available() and torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def weight_bytes_hit(w, counts_kept=None) -> int:
    """Bytes of the expert weights a forward reads: every expert that received a
    row, plus the shared expert and the router weight."""
    es = 2 if w.dtype == "bf16" else 4
    m = 3 if w.act == "silu_gated" else 2
    per_expert = m * w.d * w.h * es
    hit = w.N if counts_kept is None else int(sum(1 for c in counts_kept if c > 0))
    shared = 3 * w.d * w.h_shared * es if w.h_shared else 0
    return hit * per_expert + shared + 4 * w.d * w.N


def algorithmic(w, rows: int, counts_kept=None) -> dict:
    """Algorithmic FLOPs and bytes of one layer forward and of its expert products."""
    es = 2 if w.dtype == "bf16" else 4
    m = 3 if w.act == "silu_gated" else 2
    p1 = 2 * (m - 1) * rows * w.d * w.h + (2 * 2 * w.T * w.d * w.h_shared if w.h_shared else 0)
    p2 = 2 * rows * w.d * w.h + (2 * w.T * w.d * w.h_shared if w.h_shared else 0)
    bytes_ = weight_bytes_hit(w, counts_kept) + 2 * w.T * w.d * es
    # per-product HBM bytes: the weights of every expert that received a row, the
    # rows read and the rows written (shared expert included)
    hit = w.N if counts_kept is None else int(sum(1 for c in counts_kept if c > 0))
    hs = w.h_shared or 0
    b1 = ((m - 1) * w.d * w.h * hit + 2 * w.d * hs) * es \
        + (rows * w.d + rows * w.h) * es + ((w.T * w.d + w.T * hs) * es if hs else 0)
    b2 = (w.d * w.h * hit + w.d * hs) * es + (rows * w.h + rows * w.d) * es \
        + ((w.T * hs + w.T * w.d) * es if hs else 0)
    return {"flops": p1 + p2, "flops_p1": p1, "flops_p2": p2, "bytes": bytes_,
            "bytes_p1": b1, "bytes_p2": b2, "router_flops": 2 * w.T * w.d * w.N}


def captured_traffic(workload: str, stage: str):
    """DRAM bytes per launch of an expert-product kernel from the committed ncu
    capture (profiles/roofline_traffic.json), or None when there is none for this
    workload or the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["sources_sha256"]:
            return None
        ks = rec["workloads"][workload][stage]
        ks = ks if isinstance(ks, list) else [ks]  # a stage can be two launches (tail split)
        return sum(int(k["dram_read"]) + int(k["dram_write"]) for k in ks)
    except (OSError, KeyError, ValueError):
        return None


def router_np(N: int) -> int:
    """Experts per lane group of the N <= 32 router kernel (4, 8, 16 or 32)."""
    return 4 if N <= 4 else 8 if N <= 8 else 16 if N <= 16 else 32


def launches_per_forward(w) -> int:
    """Kernels one moe_forward launches. Token choice: router weight re-layout,
    logits with gating (one kernel for N <= 32, logits and gating kernels above),
    expert scan (folded into the slot assignment when the router has at most 32 tiles
    and N·k·tiles <= 4096 counts), slot assignment. Expert Choice: weight re-layout, logits, scores,
    per-expert selection, per-token list scan and fill, and the per-expert counts (the
    benchmark asks for them). Then
    dispatch, expert product 1 (two launches for ReLU experts with a shared expert),
    expert product 2 and the combine. With bf16 experts receiving 224 to 511 rows on
    average (the row buffers' size over N) each product is two launches: the CTA-pair
    kernel and a single-CTA kernel for the short last row blocks."""
    if w.routing == "expert_choice":
        router = 7
    else:
        tt = 64 if w.N > 32 else 4 * (32 // router_np(w.N))  # tokens per router tile
        tiles = -(-w.T // tt)
        fused_scan = tiles <= 32 and w.N * w.k * tiles <= 4096
        router = 1 + (2 if w.N > 32 else 1) + (1 if fused_scan else 2)
    p1 = 2 if (w.act == "relu" and w.h_shared) else 1
    p2 = 1
    if w.dtype == "bf16":
        if w.routing == "expert_choice":
            rows = w.N * min(-(-w.T * w.capacity_factor[0] // (w.N * w.capacity_factor[1])), w.T)
        elif w.capacity_factor:
            rows = min(w.T * w.k, w.N * -(-w.T * w.capacity_factor[0] // (w.N * w.capacity_factor[1])))
        else:
            rows = w.T * w.k
        if 224 * w.N <= rows < 512 * w.N:
            p1, p2 = p1 + 1, p2 + 1
    return router + 1 + p1 + p2 + 1


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm": float(p["hbm_gbs"]), "bf16": float(p["bf16_tflops"]),
                "bf16_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm": 6400.0, "bf16": 1800.0, "bf16_sustained": 1400.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, enabled: bool = True):
        self.idx = device_index
        self.proc = None
        self.file = None
        if enabled:
            try:
                self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.Q}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=self.file, stderr=subprocess.DEVNULL)
                time.sleep(0.3)
            except OSError:
                self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                clk, cmax = float(r[1]), float(r[2])
            except (ValueError, IndexError):
                continue
            mx = max(mx, cmax)
            sm.append(clk)
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        loaded = [c for c in sm if c > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _blas_threads() -> int:
    """Threads the oracle's float64 BLAS calls use (its C router runs on one thread):
    the pool's size as threadpoolctl reports it, else the OPENBLAS_NUM_THREADS that
    numpy's OpenBLAS read when it loaded."""
    try:
        from threadpoolctl import threadpool_info
        import numpy  # noqa: F401  (loads the BLAS so that it is listed)
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    try:
        return max(1, int(os.environ.get("OPENBLAS_NUM_THREADS", "1")))
    except ValueError:
        return 1


# ------------------------------------------------------------------ CPU oracle legs

class _HostExperts:
    """Host copy of a [N][...] weight stack, indexed per expert by the oracle."""

    def __init__(self, t, dtype):
        self.t = t.float().cpu().numpy().astype(dtype, copy=False)

    def __getitem__(self, e):
        return self.t[e]


def _oracle_inputs(inp, w):
    """Host arrays for the oracle, prepared once outside any timed region. The
    expert weights are handed over as float64 (the oracle's own precision) when
    they fit in 32 GB of host memory, else as float32 (converted per call)."""
    import numpy as np
    es = 8 if weight_bytes_hit(w) // (2 if w.dtype == "bf16" else 4) * 8 <= 32 * 2**30 else 4
    dt = np.float64 if es == 8 else np.float32
    out = {"x": inp["x"].float().cpu().numpy(), "w_r": inp["w_r"].cpu().numpy(),
           "b_r": None if inp["b_r"] is None else inp["b_r"].cpu().numpy()}
    for n in ("w_gate", "w_up", "w_down"):
        out[n] = None if inp[n] is None else _HostExperts(inp[n], dt)
    for n in ("shared_w_gate", "shared_w_up", "shared_w_down"):
        out[n] = None if inp[n] is None else inp[n].float().cpu().numpy().astype(dt)
    return out


def time_oracle(w, host_inp, sample: int, seed: int) -> tuple[float, float]:
    """One oracle pass: routing for all T tokens, outputs for `sample` tokens.
    Returns (seconds, tokens of output computed)."""
    import numpy as np
    from oracle import moe_oracle as O
    rng = np.random.default_rng(seed)
    n = min(sample, w.T)
    toks = np.sort(rng.choice(w.T, size=n, replace=False))
    t0 = time.perf_counter()
    if w.routing == "expert_choice":
        O.forward_expert_choice(w, host_inp, tokens=toks)
    else:
        O.forward(w, host_inp, tokens=toks)
    return time.perf_counter() - t0, n


class _LazyExperts:
    """Host float32 copies of the experts of a [N][...] device stack, fetched on first
    use and kept (so that a timed oracle pass finds them already in host memory)."""

    def __init__(self, t):
        self.t, self.cache = t, {}

    def __getitem__(self, e):
        if e not in self.cache:
            self.cache[e] = self.t[e].float().cpu().numpy()
        return self.cache[e]


def oracle_sample_baseline(w, inp, cpu_seconds: float) -> dict:
    """The oracle on a bounded sample of workload `w`: a batch of the first n tokens
    of the same layer (all of its steps: routing of the n tokens, their layer outputs),
    n grown until one pass takes about `cpu_seconds`. The expert weights a pass needs
    are fetched to host memory (float32) before it is timed."""
    import numpy as np
    from oracle import moe_oracle as O
    threads = _blas_threads()
    host = {"w_r": inp["w_r"].cpu().numpy(),
            "b_r": None if inp["b_r"] is None else inp["b_r"].cpu().numpy()}
    for nme in ("w_gate", "w_up", "w_down"):
        host[nme] = None if inp[nme] is None else _LazyExperts(inp[nme])
    for nme in ("shared_w_gate", "shared_w_up", "shared_w_down"):
        host[nme] = None if inp[nme] is None else inp[nme].float().cpu().numpy()
    x_all = inp["x"].float().cpu().numpy()

    ec = w.routing == "expert_choice"

    def one_pass(n):
        wn = w.replace(T=n)
        hn = dict(host, x=x_all[:n])
        if ec:  # every expert takes its top tokens
            experts = range(w.N)
        else:   # untimed: which experts to fetch
            experts = np.unique(O.route(wn, hn["x"], hn["w_r"], hn["b_r"])["topk_idx"])
        for e in experts:
            for nme in ("w_gate", "w_up", "w_down"):
                if hn[nme] is not None:
                    hn[nme][int(e)]
        t0 = time.perf_counter()
        (O.forward_expert_choice if ec else O.forward)(wn, hn)
        return time.perf_counter() - t0

    n, secs = 1, one_pass(1)
    while secs < cpu_seconds and n < w.T:
        n = min(w.T, max(n + 1, int(n * min(8.0, cpu_seconds / max(secs, 1e-3)))))
        secs = one_pass(n)
    return {"value": n / secs, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"one oracle pass over a batch of the first {n} tokens of the layer (routing and "
                      f"layer outputs of all {n}) in {secs:.4f} s; fp32 router in C on one thread, "
                      f"float64 numpy elsewhere on {threads} BLAS thread(s)"}


def run_reference(a, w, world, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = W.make_inputs(w, device=dev)
    host_inp = _oracle_inputs(inp, w)
    del inp
    sample = max(1, min(a.cpu_sample, w.T) // 4)
    for i in range(a.warmup):
        time_oracle(w, host_inp, sample, 100 + i)
    secs, toks = 0.0, 0
    for i in range(a.steps):
        s, n = time_oracle(w, host_inp, sample, 1000 + i)
        secs += s
        toks += n
    value = toks / secs
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1000 * secs / a.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "d": w.d, "N": w.N, "k": w.k, "h": w.h,
                       "h_shared": w.h_shared, "gating": w.gating, "act": w.act, "routing": w.routing,
                       "routing": w.routing},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _blas_threads(),
                             "kind": "oracle",
                             "sample": f"per step: routing of all {w.T} tokens + layer outputs "
                                       f"of {sample} random tokens (fp32 router, float64 rest)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- router variant legs

def _time_calls(fn, stream, iters: int, warmup: int = 3) -> float:
    """Mean ms of fn() over `iters` back-to-back calls, CUDA events on `stream`."""
    for _ in range(warmup):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(iters):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / iters


def measure_router_train(w, inp, cfg, ws, stream, dev, cpu_tokens: int) -> dict:
    """Training-time router (noisy top-k + z-loss) against the inference router on
    the same inputs: CUDA-event times, the logits' share of the fp32 FMA peak, and
    the oracle's training router timed on a token sample of the host cores."""
    import sparse_mixture_experts_64_b300 as moe
    T, k, N = w.T, w.k, w.N
    g = torch.Generator(device=dev).manual_seed(77)
    noise = torch.randn((T, N), device=dev, generator=g)
    i32 = dict(dtype=torch.int32, device=dev)
    o = [torch.empty((T, k), **i32), torch.empty((T, k), device=dev), torch.empty(N, **i32),
         torch.empty(N, **i32), torch.empty(N + 1, **i32), torch.empty((T, k), **i32),
         torch.empty(moe.moe_max_rows(cfg), **i32), torch.empty(2, device=dev)]
    z = torch.empty(1, device=dev)

    def infer():
        moe.moe_router_topk(cfg, inp["x"], inp["w_r"], inp["b_r"], *o, ws, stream)

    def train():
        moe.moe_router_topk_train(cfg, inp["x"], inp["w_r"], inp["b_r"], noise, 1.0, *o[:7], o[7],
                                  z, ws, stream)
    iters = 20
    ms_inf = _time_calls(infer, stream, iters)
    ms_train = _time_calls(train, stream, iters)
    st = moe.moe_check_error(ws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError("device error word: " + moe.status_str(st))
    fma_peak = 148 * 128 * 2 * 2.032e9
    flops = 2.0 * T * w.d * N
    out = {"train_ms": ms_train, "inference_ms": ms_inf, "overhead_ms": ms_train - ms_inf,
           "router_flops_fp32": flops, "bound": "alu",
           "frac": flops / (ms_train / 1e3) / fma_peak,
           "peak": "148 SMs x 128 FP32 lanes x 2 x 2032 MHz (fp32 FMA, logits only)"}
    if cpu_tokens > 0:
        from oracle import moe_oracle as O
        n = min(T, cpu_tokens)
        ws_ = w.replace(T=n)
        xs = inp["x"][:n].float().cpu().numpy()
        t0 = time.perf_counter()
        O.route_train(ws_, xs, inp["w_r"].cpu().numpy(),
                      None if inp["b_r"] is None else inp["b_r"].cpu().numpy(),
                      noise[:n].cpu().numpy(), 1.0)
        secs = time.perf_counter() - t0
        out["cpu_oracle"] = {"tokens_per_s": n / secs, "sample_tokens": n, "cores": 1,
                             "kind": "oracle"}
    return out


def measure_router_sharded(w, inp, stream, dev, cpu_tokens: int, shards: int = 2, capacity_factor=(5, 4)) -> dict:
    """GShard-style top-k with one capacity for the whole batch (factor 1.25) over the
    batch split into `shards` token shards in token order, as that many ranks would hold
    it, the shards run one after another on this GPU: phase 1 (moe_router_shard_stats:
    routing and the per-(expert, slot) statistics) per shard, the exchange's host step
    (the statistics copied to the host, the global priorities and the rank-order sums,
    the results copied back: on ranks, an all-gather), phase 2 (moe_router_shard_assign:
    the capacity decisions at the global priorities) per shard. Against moe_router_topk on
    the whole batch with the same capacity, whose kept counts the shards' must add up to
    bit for bit; the logits' share of the fp32 FMA peak; the oracle's routing timed on a
    token sample of the host cores."""
    import numpy as np

    import sparse_mixture_experts_64_b300 as moe
    from sparse_mixture_experts_64_b300 import sharded
    wg = w.replace(capacity_factor=capacity_factor)
    T, k, N = wg.T, wg.k, wg.N
    i32 = dict(dtype=torch.int32, device=dev)
    cfg_of = lambda ww: moe.make_config(**{f: getattr(ww, f) for f in ww.__dataclass_fields__})  # noqa: E731
    cuts = [T * r // shards for r in range(shards + 1)]
    sh = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        c = cfg_of(wg.replace(T=b - a, capacity_factor=None))
        sh.append(dict(a=a, b=b, cfg=c, ws=moe.workspace(c, device=dev), x=inp["x"][a:b],
                       idx=torch.empty((b - a, k), **i32), gate=torch.empty((b - a, k), device=dev),
                       cnt=torch.empty((N, k), **i32), psum=torch.empty(N, device=dev),
                       kept=torch.empty(N, **i32), off=torch.empty(N + 1, **i32),
                       slot_row=torch.empty((b - a, k), **i32),
                       perm=torch.empty(moe.moe_max_rows(c), **i32), aux=torch.empty(2, device=dev)))
    C = sharded.global_capacity(T, N, capacity_factor)
    glob = {}

    def phase1():
        for s in sh:
            moe.moe_router_shard_stats(s["cfg"], s["x"], inp["w_r"], inp["b_r"], s["idx"], s["gate"], s["cnt"],
                                       s["psum"], s["ws"], stream)

    def exchange():
        counts = np.stack([s["cnt"].cpu().numpy() for s in sh])
        bases = sharded.slot_bases(counts)
        psum = np.zeros(N, np.float32)
        for s in sh:  # rank order
            psum = (psum + s["psum"].cpu().numpy()).astype(np.float32)
        glob["routed"] = torch.as_tensor(counts.sum(axis=(0, 2)), dtype=torch.int32).to(dev)
        glob["psum"] = torch.as_tensor(psum).to(dev)
        for r, s in enumerate(sh):
            s["base"] = torch.as_tensor(bases[r], dtype=torch.int32).to(dev)
        torch.cuda.synchronize()

    def phase2():
        for s in sh:
            moe.moe_router_shard_assign(s["cfg"], s["idx"], s["base"], C, glob["routed"], glob["psum"], T, s["kept"],
                                        s["off"], s["slot_row"], s["perm"], s["aux"], s["ws"], stream)
    iters = 20
    ms1 = _time_calls(phase1, stream, iters) / shards
    torch.cuda.synchronize()
    host = []
    for _ in range(iters):
        t0 = time.perf_counter()
        exchange()
        host.append((time.perf_counter() - t0) * 1e3)
    ms2 = _time_calls(phase2, stream, iters) / shards
    # the whole batch with the same capacity on one router call
    cw = cfg_of(wg)
    ws_w = moe.workspace(cw, device=dev)
    o = [torch.empty((T, k), **i32), torch.empty((T, k), device=dev), torch.empty(N, **i32), torch.empty(N, **i32),
         torch.empty(N + 1, **i32), torch.empty((T, k), **i32), torch.empty(moe.moe_max_rows(cw), **i32),
         torch.empty(2, device=dev)]
    ms_w = _time_calls(lambda: moe.moe_router_topk(cw, inp["x"], inp["w_r"], inp["b_r"], *o, ws_w, stream),
                       stream, iters)
    for s in sh + [dict(ws=ws_w)]:
        st = moe.moe_check_error(s["ws"], stream)
        if st != moe.MOE_OK:
            raise RuntimeError("device error word: " + moe.status_str(st))
    kept_shards = sum(s["kept"].cpu().numpy().astype(np.int64) for s in sh)
    if not np.array_equal(kept_shards, o[3].cpu().numpy()):
        raise RuntimeError("sharded capacity decisions differ from the whole batch's")
    ms_x = statistics.median(host)
    fma_peak = 148 * 128 * 2 * 2.032e9
    flops = 2.0 * (T // shards) * w.d * N
    out = {"shards": shards, "capacity_factor": list(capacity_factor), "capacity": C, "top_k": k,
           "phase1_ms_per_shard": ms1, "exchange_host_ms": ms_x, "phase2_ms_per_shard": ms2,
           "rank_ms": ms1 + ms_x + ms2, "tokens_per_s_per_rank": (T / shards) / ((ms1 + ms_x + ms2) / 1e3),
           "whole_batch_router_ms": ms_w, "kept_counts_equal_whole_batch": True,
           "dropped_slots": int(T * k - int(kept_shards.sum())), "bound": "alu",
           "frac": flops / (ms1 / 1e3) / fma_peak,
           "peak": "148 SMs x 128 FP32 lanes x 2 x 2032 MHz (fp32 FMA, phase 1's logits)",
           "exchange": "host step standing in for the all-gather of N x k counts and N sums per rank"}
    if cpu_tokens > 0:
        from oracle import moe_oracle as O
        n = min(T, cpu_tokens)
        xs = inp["x"][:n].float().cpu().numpy()
        t0 = time.perf_counter()
        O.route(wg.replace(T=n), xs, inp["w_r"].cpu().numpy(),
                None if inp["b_r"] is None else inp["b_r"].cpu().numpy())
        secs = time.perf_counter() - t0
        out["cpu_oracle"] = {"tokens_per_s": n / secs, "sample_tokens": n, "cores": 1, "kind": "oracle"}
    return out


def measure_backward(w, inp, cfg, ws, stream, dev, peaks, host_inp=None, cpu_tokens: int = 16) -> dict:
    """The training step's backward: moe_forward with save_preact (it keeps the experts'
    pre-activations) and moe_backward on the same inputs. CUDA-event times of the
    backward alone, of the keeping forward alone and of the pair back to back; the
    backward's algorithmic FLOPs (the gradient products: dH, dX and the weight gradients
    of the experts and the shared expert, and the router's two) against the bf16 peak;
    the backward that recomputes the pre-activations (plain forward) for comparison; and
    the oracle's backward timed on a token slice of the same layer."""
    import sparse_mixture_experts_64_b300 as moe
    T, d, N, k = w.T, w.d, w.N, w.k
    keep_cfg = moe.make_config(**{f: getattr(w, f) for f in w.__dataclass_fields__}, save_preact=True)
    ws_keep = moe.workspace(keep_cfg, device=dev)
    bws = moe.backward_workspace(cfg, device=dev)  # the larger one: it holds recomputed pre-activations
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gate = torch.empty((T, k), device=dev)
    y = torch.empty((T, d), dtype=inp["x"].dtype, device=dev)
    kept = torch.empty(N, dtype=torch.int32, device=dev)

    def fwd(c, wsp):
        moe.moe_forward(c, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"],
                        inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"], y, idx, gate, None, kept,
                        None, wsp, stream)
    g = torch.Generator(device=dev).manual_seed(17)
    dy = torch.randn((T, d), device=dev, generator=g).to(inp["x"].dtype)
    e = lambda t: None if t is None else torch.empty_like(t)  # noqa: E731
    out = [e(inp["x"]), e(inp["w_r"]), e(inp["b_r"]), e(inp["w_gate"]), e(inp["w_up"]), e(inp["w_down"]),
           e(inp["shared_w_gate"]), e(inp["shared_w_up"]), e(inp["shared_w_down"])]

    def bwd(c, wsp):
        moe.moe_backward(c, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"],
                         inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"], idx, gate, dy, 0.01, 0.001,
                         *out, wsp, bws, stream)
    fwd(cfg, ws)
    ms_recompute = _time_calls(lambda: bwd(cfg, ws), stream, 10)
    fwd(keep_cfg, ws_keep)
    ms = _time_calls(lambda: bwd(keep_cfg, ws_keep), stream, 10)
    fwd_keep_ms = _time_calls(lambda: fwd(keep_cfg, ws_keep), stream, 10)
    fwd_plain_ms = _time_calls(lambda: fwd(cfg, ws), stream, 10)  # the same launches without keeping
    step_ms = _time_calls(lambda: (fwd(keep_cfg, ws_keep), bwd(keep_cfg, ws_keep)), stream, 10)
    for wsp in (ws, ws_keep):
        st = moe.moe_check_error(wsp, stream)
        if st != moe.MOE_OK:
            raise RuntimeError("device error word: " + moe.status_str(st))
    R = int(kept.sum().item())
    gated = w.act == "silu_gated"
    # dH (2 R d h), dX (4 R d h gated, else 2), the weight gradients (6 or 4 R d h); the
    # shared expert's 12 T d h_shared; the router's dx and dW_r (2 T d N each)
    per = 12 if gated else 8
    flops = per * R * d * w.h + (12 * T * d * w.h_shared if w.h_shared else 0) + 2 * 2 * T * d * N
    tf = lambda m: flops / (m / 1e3) / 1e12  # noqa: E731
    out_d = {"ms": ms, "tokens_per_s": T / (ms / 1e3), "rows": R, "algorithmic_flops": flops,
             "achieved_tflops": tf(ms), "bound": "tensor", "frac": tf(ms) / peaks["bf16"],
             "peak": f"{peaks['source']} bf16 burst {peaks['bf16']} TFLOP/s",
             "pre_activations": "kept by the forward (save_preact)",
             "forward_keeping_ms": fwd_keep_ms, "forward_plain_ms": fwd_plain_ms,
             "forward_plus_backward_ms": step_ms,
             "recompute": {"ms": ms_recompute, "achieved_tflops": tf(ms_recompute),
                           "frac": tf(ms_recompute) / peaks["bf16"],
                           "note": "plain forward; the backward recomputes the pre-activations "
                                   "(not counted as algorithmic FLOPs)"}}
    if host_inp is not None:
        from oracle import moe_oracle as O
        n = min(T, cpu_tokens)
        wn = w.replace(T=n)
        host = dict(host_inp, x=host_inp["x"][:n])
        t0 = time.perf_counter()
        O.backward(wn, host, dy[:n].float().cpu().numpy(), aux_coef=0.01, z_coef=0.001)
        secs = time.perf_counter() - t0
        out_d["cpu_oracle"] = {"tokens_per_s": n / secs, "sample_tokens": n, "cores": _blas_threads(),
                               "kind": "oracle"}
    return out_d


# ------------------------------------------------------------------------ GPU arm

def measure(a, w, world, rank, local, primary: bool = True) -> dict:
    """Time the layer forward of workload `w` (the bench contract's step) and return its
    JSON record. primary: the headline workload, with the router/backward variants and
    the full oracle baseline; otherwise a bounded oracle sample and no variants."""
    import sparse_mixture_experts_64_b300 as moe

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = W.make_inputs(w, device=dev)
    cfg = moe.make_config(T=w.T, d=w.d, N=w.N, k=w.k, h=w.h, h_shared=w.h_shared, dtype=w.dtype,
                          gating=w.gating, act=w.act, capacity_factor=w.capacity_factor,
                          router_bias=w.router_bias, routing=w.routing)
    ws = moe.workspace(cfg, device=dev)
    ec = w.routing == "expert_choice"
    T, k, N, d = w.T, w.k, w.N, w.d
    y = torch.empty((T, d), dtype=inp["x"].dtype, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gate = torch.empty((T, k), dtype=torch.float32, device=dev)
    routed = torch.empty(N, dtype=torch.int32, device=dev)
    kept = torch.empty(N, dtype=torch.int32, device=dev)
    aux = torch.empty(2, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    if ec:  # Expert Choice returns no token-choice outputs
        idx = gate = aux = None

    def fwd(x=None, y_out=None):
        moe.moe_forward(cfg, inp["x"] if x is None else x, inp["w_r"], inp["b_r"], inp["w_gate"],
                        inp["w_up"], inp["w_down"], inp["shared_w_gate"], inp["shared_w_up"],
                        inp["shared_w_down"], y if y_out is None else y_out, idx, gate, routed, kept, aux,
                        ws, stream)

    # L2: weights larger than L2 stream from HBM every step; otherwise flush.
    wbytes = weight_bytes_hit(w)
    flush = None
    if wbytes < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    l2_mode = ("inputs larger than L2 (%.2f GB of expert weights)" % (wbytes / 1e9) if flush is None
               else "L2 flushed between steps (256 MB write, outside the timed events)")

    for _ in range(max(3, a.warmup)):
        fwd()
    torch.cuda.synchronize(dev)
    st = moe.moe_check_error(ws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError("device error word: " + moe.status_str(st))
    counts_kept = kept.cpu().tolist()
    rows = int(sum(counts_kept))

    # ---- the forward captured once as a CUDA graph (moe_forward_graph_create); each
    # timed step launches it. Stage times come from graphs that also record six events
    # at the stage boundaries, one per step, launched between the timed steps so that
    # both run under the same clocks and power state (an event between two kernels
    # orders them fully, so those launches show each stage alone, without the
    # programmatic-launch overlap of neighbouring kernels that the timed graph has).
    def make_graph(events=None, x=None, y_out=None):
        return moe.moe_forward_graph_create(cfg, inp["x"] if x is None else x, inp["w_r"], inp["b_r"], inp["w_gate"],
                                            inp["w_up"], inp["w_down"], inp["shared_w_gate"], inp["shared_w_up"],
                                            inp["shared_w_down"], y if y_out is None else y_out, idx, gate, routed,
                                            kept, aux, ws, events=events)

    graph, pgs, graph_note = None, [], None
    try:
        graph = make_graph()
        for _ in range(a.steps):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
            for ev in evs:
                ev.record(stream)
            pgs.append((make_graph(events=evs), evs))
        for _ in range(max(3, a.warmup)):
            graph.launch(stream)
        for g_, _ in pgs[:3]:
            g_.launch(stream)
        torch.cuda.synchronize(dev)
    except (RuntimeError, moe.MoeError) as exc:
        graph_note = f"stream launches of moe_forward (graph capture failed: {exc})"
        graph, pgs = None, []

    # ---- timed region: K forwards, per-step CUDA events on the launching stream
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    clocks = ClockSampler(local, enabled=not a.no_clocks)
    _barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(a.steps):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        if graph is not None:
            graph.launch(stream)
        else:
            fwd()
        ends[i].record(stream)
        if pgs:
            if flush is not None:
                flush.zero_()
            pgs[i][0].launch(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    _barrier(world)
    clk = clocks.stop()
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / a.steps
    ms_max = _max_over_ranks(ms, world)
    value = world * T / (ms_max / 1e3)
    st = moe.moe_check_error(ws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError("device error word: " + moe.status_str(st))
    stage_from_graphs = bool(pgs)
    if pgs:
        stage_ms = [sum(e_[j].elapsed_time(e_[j + 1]) for _, e_ in pgs) / len(pgs) for j in range(5)]
        for g_, _ in pgs:
            g_.destroy()
    else:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        for ev in evs:
            ev.record(stream)
        stage_ms = [0.0] * 5
        nprof = max(10, a.steps // 2)
        for i in range(nprof):
            if flush is not None:
                flush.zero_()
            moe.moe_forward_profiled(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"],
                                     inp["w_down"], inp["shared_w_gate"], inp["shared_w_up"],
                                     inp["shared_w_down"], y, idx, gate, routed, kept, aux, ws, evs,
                                     stream)
            evs[-1].synchronize()
            for j in range(5):
                stage_ms[j] += evs[j].elapsed_time(evs[j + 1]) / nprof

    # ---- the same forwards as plain stream launches (moe_forward per step), for comparison
    for i in range(a.steps):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        fwd()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    stream_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / a.steps
    use_graph = graph is not None
    e2e_graph_src = graph

    # ---- end to end: every step copies its x from pinned host memory, runs the
    # forward and copies its y back; the copies of neighbouring steps overlap the
    # forward (double-buffered device x / y, host-to-device and device-to-host copies
    # each on their own stream, ordered by events)
    x_host = inp["x"].cpu().pin_memory()
    y_host = [torch.empty_like(y, device="cpu").pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(inp["x"]) for _ in range(2)]
    y_dev = [torch.empty_like(y) for _ in range(2)]
    e2e_graphs = [make_graph(x=x_dev[b], y_out=y_dev[b]) for b in range(2)] if use_graph else []
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("h2d", "comp", "d2h")}
    for n in ev:
        for e_ in ev[n]:
            e_.record(stream)

    def e2e_steps(n):
        for i in range(n):
            b = i & 1
            s_h2d.wait_event(ev["comp"][b])          # x_dev[b] no longer read
            with torch.cuda.stream(s_h2d):
                x_dev[b].copy_(x_host, non_blocking=True)
            ev["h2d"][b].record(s_h2d)
            stream.wait_event(ev["h2d"][b])
            stream.wait_event(ev["d2h"][b])           # y_dev[b] no longer read
            if e2e_graphs:
                e2e_graphs[b].launch(stream)
            else:
                fwd(x_dev[b], y_dev[b])
            ev["comp"][b].record(stream)
            s_d2h.wait_event(ev["comp"][b])
            with torch.cuda.stream(s_d2h):
                y_host[b].copy_(y_dev[b], non_blocking=True)
            ev["d2h"][b].record(s_d2h)
    e2e_steps(4)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ne2e = max(10, a.steps // 2)
    e0.record(s_h2d)
    stream.wait_event(e0)
    s_d2h.wait_event(e0)
    e2e_steps(ne2e)
    e1.record(s_d2h)
    torch.cuda.synchronize(dev)
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1) / ne2e, world)
    e2e_value = world * T / (e2e_ms / 1e3)
    st = moe.moe_check_error(ws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError("device error word: " + moe.status_str(st))
    for g_ in e2e_graphs:
        g_.destroy()
    if e2e_graph_src is not None:
        e2e_graph_src.destroy()

    # ---- roofline of the dominant kernel
    alg = algorithmic(w, rows, counts_kept)
    peaks = _peaks()
    stage = dict(zip(STAGES, stage_ms))
    if w.dtype == "bf16":
        dom = max(("expert_product_1", "expert_product_2"), key=lambda s: stage[s])
        p = "1" if dom == "expert_product_1" else "2"
        flops, nbytes = alg["flops_p" + p], alg["bytes_p" + p]
        sec = stage[dom] / 1e3
        traffic = captured_traffic(w.name, dom)
        kind = ("gated" if w.act == "silu_gated" else "relu") if p == "1" else "plain"
        kernel = f"expert product {p}: k_ffn_tc2<{kind}> (CTA pair) or k_ffn_tc<{kind}>"
        # the kernel's bound is whichever floor is higher: its FLOPs at the tensor
        # peak or its bytes at the HBM peak
        if nbytes / (peaks["hbm"] * 1e9) > flops / (peaks["bf16"] * 1e12):
            achieved = nbytes / sec / 1e9
            roof = {"kernel": kernel, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm"], "traffic": traffic,
                    "peak_source": peaks["source"] + " HBM copy"}
        else:
            achieved = flops / sec / 1e12
            roof = {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": peaks["bf16"],
                    "unit": "TFLOP/s", "frac": achieved / peaks["bf16"], "traffic": traffic,
                    "peak_source": peaks["source"] + " bf16 burst",
                    # the kernel runs inside back-to-back steps under the power cap, where
                    # the sustained figure (a seconds-long cuBLAS loop) is the comparable one
                    "frac_of_sustained_peak": achieved / peaks["bf16_sustained"],
                    "sustained_peak": peaks["bf16_sustained"]}
        roof.update({"algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": nbytes,
                     "traffic_over_algorithmic": None if traffic is None else traffic / nbytes,
                     "avg_launch_ms": stage[dom]})
    else:
        dom = "expert_product_1"
        flops = alg["flops_p1"]
        achieved = flops / (stage[dom] / 1e3) / 1e12
        fp32_peak = 148 * 128 * 2 * 2.032e9 / 1e12
        roof = {"kernel": "k_ffn_simt<gated>", "bound": "alu", "achieved": achieved,
                "peak": fp32_peak, "unit": "TFLOP/s", "frac": achieved / fp32_peak,
                "traffic": None, "peak_source": "148 SMs x 128 FP32 lanes x 2 x 2032 MHz",
                "algorithmic_flops_per_launch": flops, "avg_launch_ms": stage[dom]}
    layer_roof_ms = max(alg["flops"] / (peaks["bf16"] * 1e12), alg["bytes"] / (peaks["hbm"] * 1e9)) * 1e3

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded normal inputs and weights)",
        "config": {"workload": w.name, "T": T, "d": d, "N": N, "k": k, "h": w.h,
                   "h_shared": w.h_shared, "gating": w.gating, "act": w.act,
                   "capacity_factor": w.capacity_factor, "router": "fp32",
                   "global_batch_tokens": world * T, "parallelism": f"replicas x{world}",
                   "l2": l2_mode,
                   "launch": graph_note or "the forward as one CUDA graph per step (moe_forward_graph_launch); "
                                           "stage times from graphs with stage events launched between "
                                           "the timed steps"},
        "roofline": roof,
        "layer_roofline": {"roofline_ms": layer_roof_ms, "frac": layer_roof_ms / ms_max,
                           "algorithmic_flops": alg["flops"], "algorithmic_bytes": alg["bytes"],
                           "router_flops_fp32": alg["router_flops"],
                           "peaks": f"{peaks['source']}: bf16 {peaks['bf16']} TFLOP/s, "
                                    f"HBM {peaks['hbm']} GB/s"},
        "stages_ms": stage, "rows_dispatched": rows,
        "stream_launch_ms_per_step": stream_ms,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
                "d2h_bytes_per_step": y_host[0].numel() * y_host[0].element_size(),
                "ms_per_step": e2e_ms,
                "pipelining": "copies of neighbouring steps overlap the forward (2 buffers, 3 streams)",
                "launch": "moe_forward_graph_launch" if e2e_graphs else "moe_forward"},
        # each timed step launches the forward graph and, between steps, one
        # stage-event graph of the same kernels
        "gpu_launches": launches_per_forward(w) * a.steps * (2 if stage_from_graphs else 1),
        "clocks": clk, "wall_s_timed": wall,
        # expert weights that received rows (+ shared + router) per forward, over the step time
        "weight_stream_gbs": weight_bytes_hit(w, counts_kept) / (ms_max / 1e3) / 1e9,
    }

    # ---- training-time router variant (noisy top-k + z-loss), same inputs
    cpu = rank == 0 and world == 1 and not a.no_cpu_baseline
    host_inp = _oracle_inputs(inp, w) if cpu and primary else None
    if primary and not a.no_variants and not ec:
        line["variants"] = {"router_train": measure_router_train(w, inp, cfg, ws, stream, dev, 512 if cpu else 0),
                            "router_sharded": measure_router_sharded(w, inp, stream, dev, 512 if cpu else 0)}
        if w.dtype == "bf16":
            line["variants"]["backward"] = measure_backward(w, inp, cfg, ws, stream, dev, peaks, host_inp)
    elif not primary and not a.no_variants and w.name == "deepseek_fine":
        # the backward of the fine-grained layer as well (its oracle too slow to time beside it)
        line["variants"] = {"backward": measure_backward(w, inp, cfg, ws, stream, dev, peaks, None)}

    # ---- CPU oracle baseline (rank 0, single process only)
    if cpu and not primary:
        line["cpu_baseline"] = oracle_sample_baseline(w, inp, a.secondary_cpu_seconds)
    elif cpu:
        # passes of the oracle (each: routing of all tokens, outputs of a new random
        # sample) until about --cpu-seconds of CPU time, at most 200 passes
        secs, n, passes = 0.0, 0, 0
        while passes < 200 and (passes == 0 or secs < a.cpu_seconds):
            s_, n_ = time_oracle(w, host_inp, a.cpu_sample, 7 + passes)
            secs, n, passes = secs + s_, n + n_, passes + 1
        line["cpu_baseline"] = {
            "value": n / secs, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{passes} pass(es), each routing all {T} tokens and computing the layer outputs of "
                      f"{min(a.cpu_sample, T)} random tokens: {n} outputs in {secs:.1f} s "
                      f"(fp32 router in C on one thread, float64 numpy elsewhere on "
                      f"{_blas_threads()} BLAS thread(s))"}
    return line


def _summary(sub: dict) -> dict:
    """The fields of a secondary workload's record kept in the headline line."""
    keep = ("value", "unit", "ms_per_step", "dtype", "config", "layer_roofline", "stages_ms",
            "weight_stream_gbs", "rows_dispatched", "gpu_launches", "clocks", "cpu_baseline", "e2e",
            "stream_launch_ms_per_step", "variants")
    out = {k: sub[k] for k in keep if k in sub}
    r = sub["roofline"]
    out["roofline"] = {k: r[k] for k in ("kernel", "bound", "achieved", "peak", "unit", "frac", "traffic",
                                         "peak_source", "avg_launch_ms", "algorithmic_flops_per_launch",
                                         "algorithmic_bytes_per_launch", "traffic_over_algorithmic")
                       if k in r}
    return out


def run_ours(a, w, world, rank, local, secondary: bool):
    line = measure(a, w, world, rank, local, primary=True)
    if secondary:
        import gc
        line["workloads"] = {}
        for name in SECONDARY:
            if name == w.name:
                continue
            gc.collect()
            torch.cuda.empty_cache()
            line["workloads"][name] = _summary(measure(a, W.WORKLOADS[name], world, rank, local, primary=False))
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    a = _args()
    world, rank, local = _dist()
    w = W.WORKLOADS[a.config]
    over = {k: v for k, v in (("T", a.tokens), ("N", a.experts), ("h", a.hidden)) if v}
    if over:
        w = w.replace(name=w.name + "_" + "_".join(f"{k}{v}" for k, v in over.items()), **over)
    if a.impl == "reference":
        run_reference(a, w, world, rank)
    else:
        # the other workloads join the default run on one GPU (a scaling run times the
        # default workload alone)
        secondary = a.workloads == "all" or (a.workloads == "auto" and a.config == "mixtral_prefill"
                                             and not over and world == 1)
        run_ours(a, w, world, rank, local, secondary)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
