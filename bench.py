#!/usr/bin/env python3
"""Benchmark of the TurboQuant KV-cache hot path on GB300.

One step = the whole per-layer decode path for one batch: quantize-append of
each sequence's new K/V token into the packed 3-bit cache, then decode
attention of every query head over the full packed context (query prep,
split-K attention, merge + back-rotation).  Default workload: Llama-3-8B-shaped
decode layer (batch 16, 32 query heads, 8 KV heads, d 128, context 8192,
3-bit K = 2-bit MSE + 1-bit QJL, 3-bit V), synthetic bf16 K/V with
log-uniform per-channel scales and 2% outlier channels.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on the host cores on the same workload (bounded sample per step).
Multi-GPU: one process per GPU under torchrun; every rank runs its own
replica (different seeds: weak scaling, no data-path collective); the step
time is the max over ranks.
"""
import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 10 ** 6
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
METRIC = "decode attention tokens/s over the packed 3-bit KV cache"


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="c2_llama3_8b_decode")
    p.add_argument("--cpu-groups", type=int, default=48, help="oracle (sequence, KV head) groups timed")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    return p.parse_args(argv)


# ----------------------------------------------------------- ranks (host) --

def rank_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_ranks(backend):
    import torch.distributed as dist
    rank, world, _ = rank_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value, device="cpu"):
    """Max of a float over all ranks (identity with one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base, rank):
    """Each rank decodes its own sequences (independent replica)."""
    return base + 1000 * rank


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.splitlines():
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hw_thermal=parts[6], sw_thermal=parts[7], sw_power=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        idle = min(r["power"] for r in rows)
        busy = [r for r in rows if r["power"] > idle + 50] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(busy)}


# ------------------------------------------------------- roofline inputs --

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Burst bf16 dense tensor TFLOP/s (a kernel timed alone), measured or fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def measure_prefill_quantize(steps, warmup):
    """Secondary figure: quantize-append throughput of a prefill of 32768 tokens
    x 8 KV heads (bf16, 3-bit keys = 2 MSE bits + QJL, 3-bit values), two
    input copies rotated so the 128 MB of inputs are read from HBM."""
    import numpy as np
    import torch

    from online_kv_cache_tq_gb300 import binding as B
    from online_kv_cache_tq_gb300 import cache as C
    from online_kv_cache_tq_gb300 import workloads as W
    cfg = W.CONFIGS["c3_prefill_quantize"]
    n_tok, n_kv = cfg["tokens"], cfg["n_kv"]
    book = B.Codebook(k_bits=3, v_bits=3, qjl_m=cfg["qjl_m"], seed=cfg["seed"], block_size=cfg["block_size"],
                      device=torch.cuda.current_device())
    g = torch.Generator(device="cuda")
    g.manual_seed(cfg["seed"])
    inputs = [(W.student_t_tokens(n_tok, n_kv, cfg["student_t_channels"], torch.bfloat16, "cuda", g, 2 * i),
               W.student_t_tokens(n_tok, n_kv, cfg["student_t_channels"], torch.bfloat16, "cuda", g, 2 * i + 1))
              for i in range(2)]
    cache = C.allocate_cache(book, n_tok // cfg["block_size"], n_kv)
    view = C.cache_view(book, cache)
    slots = torch.arange(n_tok, device="cuda", dtype=torch.int64)

    def append(i):
        k, v = inputs[i % 2]
        B.tq_quantize_append(book, k, v, B.TQ_BF16, n_tok, n_kv, slots, view)

    for i in range(warmup):
        append(i)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record()
    for i in range(steps):
        append(i)
    end.record()
    torch.cuda.synchronize()
    if B.tq_get_last_device_error(book):
        raise RuntimeError("device error during the prefill quantize measurement")
    secs = start.elapsed_time(end) * 1e-3 / steps
    vectors = 2 * n_tok * n_kv
    field = C.cache_bytes_per_token_head(book)
    nbytes = vectors * 256 + n_tok * n_kv * field            # bf16 reads + packed writes
    flops = n_tok * n_kv * (2 * 32768) + n_tok * n_kv * 32768  # K: rotation + QJL, V: rotation
    hbm, _ = hbm_peak()
    tensor, tensor_src = bf16_peak()
    rec = [recorded_traffic(k, "c3_prefill_quantize") for k in ("quantize_tc_kernel<2,1,0>", "quantize_tc_kernel<3,0,1>")]
    traffic = sum(rec) if all(r is not None for r in rec) else None
    return {"workload": "c3_prefill_quantize", "tokens": n_tok, "n_kv_heads": n_kv, "k_bits": 3, "v_bits": 3,
            "ms_per_append": secs * 1e3, "vectors_per_s": vectors / secs,
            "hbm_gbs": nbytes / secs / 1e9, "hbm_frac": nbytes / secs / 1e9 / hbm,
            "algorithmic_tflops": flops / secs / 1e12, "tensor_frac": flops / secs / 1e12 / tensor,
            "tensor_peak": tensor, "tensor_peak_source": tensor_src + " bf16_tflops",
            "algorithmic_bytes_per_append": nbytes, "traffic_bytes_per_append": traffic,
            "note": "algorithmic flops; the bf16 hi/lo splitting runs 2 (rotation) and 3 (QJL) tensor passes"}


def source_digest(rel):
    with open(os.path.join(ROOT, rel), "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch of ``kernel`` from the committed ncu summary, or
    None when absent or taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "kernel_traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)[workload][kernel]
        if rec.get("source_sha256") != source_digest(rec["source"]):
            return None
    except (OSError, KeyError, ValueError):
        return None
    return rec.get("dram_bytes_per_launch")


# --------------------------------------------------------- decode (ours) --

class DecodeWorkload:
    """Packed caches (several copies when one fits in L2), new-token K/V and
    queries of one decode workload, resident in HBM."""

    def __init__(self, name, device, seed):
        import numpy as np
        import torch

        from online_kv_cache_tq_gb300 import binding as B
        from online_kv_cache_tq_gb300 import cache as C
        from online_kv_cache_tq_gb300 import workloads as W
        self.B, self.C, self.np, self.torch = B, C, np, torch
        cfg = W.CONFIGS[name]
        self.cfg = cfg
        self.name = name
        self.batch, self.n_q, self.n_kv = cfg["batch"], cfg["n_q"], cfg["n_kv"]
        self.book = B.Codebook(k_bits=cfg["k_bits"], v_bits=cfg["v_bits"], qjl_m=cfg["qjl_m"], seed=cfg["seed"],
                               block_size=cfg["block_size"], device=device)
        self.ctx = W.context_lengths(cfg, seed)
        self.max_ctx = int(self.ctx.max())
        self.table, num_blocks = W.block_layout(self.ctx, cfg["block_size"], cfg.get("shuffled_table", False), seed)
        self.max_blocks = self.table.shape[1]
        dt = W.torch_dtype(cfg["dtype"])
        self.dtype_code = B.TQ_BF16 if dt == torch.bfloat16 else B.TQ_FP32
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        prof = (cfg.get("log_uniform"), cfg.get("outliers", 0), cfg.get("outlier_scale", 1.0))
        ks = W.channel_scales(seed, self.n_kv, *prof)
        vs = W.channel_scales(seed + 1, self.n_kv, *prof)
        base = C.allocate_cache(self.book, num_blocks, self.n_kv)
        view = C.cache_view(self.book, base)
        bs = cfg["block_size"]
        for b, length in enumerate(self.ctx):
            for s0 in range(0, int(length) - 1, 8192):
                n = min(8192, int(length) - 1 - s0)
                k = W.gaussian_tokens(n, ks, dt, "cuda", g)
                v = W.gaussian_tokens(n, vs, dt, "cuda", g)
                slots = torch.as_tensor(W.slots_for(self.table[b], np.arange(s0, s0 + n), bs), device="cuda")
                B.tq_quantize_append(self.book, k, v, self.dtype_code, n, self.n_kv, slots, view)
        self.bytes_per_token_head = C.cache_bytes_per_token_head(self.book)
        self.cache_bytes = int(self.ctx.sum()) * self.n_kv * self.bytes_per_token_head
        copies = 1 if self.cache_bytes > 2 * L2_BYTES else math.ceil(2 * L2_BYTES / self.cache_bytes) + 1
        self.caches = [base] + [{n: t.clone() for n, t in base.items()} for _ in range(copies - 1)]
        self.views = [C.cache_view(self.book, c) for c in self.caches]
        # the step's inputs: one new K/V token per sequence (at position ctx-1) and the queries
        self.k_new = W.gaussian_tokens(self.batch, ks, dt, "cuda", g)
        self.v_new = W.gaussian_tokens(self.batch, vs, dt, "cuda", g)
        self.q = W.queries(self.batch, self.n_q, dt, "cuda", g)
        self.table_d = torch.as_tensor(self.table, device="cuda")
        self.ctx_d = torch.as_tensor(self.ctx, device="cuda")
        self.out = torch.empty((self.batch, self.n_q, 128), dtype=torch.float32, device="cuda")
        self.ws, self.ws_bytes = C.allocate_workspace(self.book, self.batch, self.n_q, self.max_ctx)
        torch.cuda.synchronize()
        # tq_decode_step: append + query preparation (one launch up to 1024 head vectors, else
        # quantize K, quantize V, prepare), partials, merge
        self.launches_per_step = (1 if self.batch * self.n_kv <= 1024 else 3) + 2

    def step(self, i):
        """One decode step: tq_decode_step (append the new K/V token of every
        sequence, then decode attention), inputs resident on the device."""
        self.B.tq_decode_step(self.book, self.k_new, self.v_new, self.dtype_code, self.q, self.dtype_code,
                              self.batch, self.n_q, self.n_kv, self.views[i % len(self.views)], self.table_d,
                              self.max_blocks, self.ctx_d, self.max_ctx, 0.0, self.out, self.ws, self.ws_bytes)

    def staged_step(self, i, ev):
        """The same step through the staged calls (same kernels, without the
        early start of the partials kernel), with events around the partials."""
        B = self.B
        view = self.views[i % len(self.views)]
        B.tq_decode_step_prepare(self.book, self.k_new, self.v_new, self.dtype_code, self.q, self.dtype_code,
                                 self.batch, self.n_q, self.n_kv, view, self.table_d, self.max_blocks, self.ctx_d,
                                 self.max_ctx, self.ws, self.ws_bytes)
        if ev is not None:
            ev[0].record()
        B.tq_decode_partials(self.book, self.batch, self.n_q, self.n_kv, view, self.table_d, self.max_blocks,
                             self.ctx_d, self.max_ctx, 0.0, self.ws, self.ws_bytes)
        if ev is not None:
            ev[1].record()
        B.tq_decode_finish(self.book, self.batch, self.n_q, self.ctx_d, self.max_ctx, self.max_blocks, self.out,
                           self.ws, self.ws_bytes)

    def e2e(self, steps, warmup):
        """Same step through the one-call C entry point for host buffers
        (tq_decode_step_host): per step the H2D copies of the step's inputs
        from pinned host memory, the step, the D2H copy of the output, and a
        synchronisation before the host reads it."""
        torch, B = self.torch, self.B
        host = {name: t.cpu().pin_memory() for name, t in
                (("q", self.q), ("k", self.k_new), ("v", self.v_new), ("ctx", self.ctx_d))}
        out_h = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        ws_bytes = B.tq_decode_step_host_workspace_bytes(self.book, self.batch, self.n_q, self.n_kv, self.max_ctx,
                                                         self.dtype_code, self.dtype_code)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_h.numel() * out_h.element_size()
        stream = torch.cuda.current_stream()

        def one(i):
            view = self.views[i % len(self.views)]
            B.tq_decode_step_host(self.book, host["k"], host["v"], self.dtype_code, host["q"], self.dtype_code,
                                  self.batch, self.n_q, self.n_kv, view, self.table_d, self.max_blocks, host["ctx"],
                                  self.max_ctx, 0.0, out_h, ws, ws_bytes, stream)
            stream.synchronize()

        for i in range(warmup):
            one(i)
        t0 = time.perf_counter()
        for i in range(steps):
            one(i)
        return time.perf_counter() - t0, h2d, d2h


def run_ours(args, rank, world, local_rank):
    import torch
    torch.cuda.set_device(local_rank)
    import __graft_entry__
    __graft_entry__.build()
    wl = DecodeWorkload(args.workload, local_rank, rank_seed(0, rank))
    for i in range(args.warmup):
        wl.step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    start.record()
    for i in range(args.steps):
        wl.step(args.warmup + i)
    end.record()
    torch.cuda.synchronize()
    barrier()
    # the dominant kernel's duration: the same steps through the staged calls,
    # with events around each partials launch on the launching stream
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        wl.staged_step(args.warmup + args.steps + i, events[i])
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    total_ms = start.elapsed_time(end)
    attn_ms = sum(a.elapsed_time(b) for a, b in events) / args.steps
    err = wl.B.tq_get_last_device_error(wl.book)
    if err:
        raise RuntimeError("device error %d during the benchmark" % err)
    dev = "cuda" if world > 1 else "cpu"
    max_ms = max_over_ranks(total_ms, dev)
    max_attn = max_over_ranks(attn_ms, dev)
    quant = measure_prefill_quantize(20, 3)
    e2e = None
    if not args.no_e2e:
        secs, h2d, d2h = wl.e2e(args.steps, min(args.warmup, 5))
        secs = max_over_ranks(secs, dev)
        e2e = {"value": world * wl.batch * args.steps / secs, "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    return wl, max_ms, max_attn, clock_info, e2e, quant


# ----------------------------------------------------- oracle (reference) --

def _oracle_group(task):
    """Oracle time for one (sequence, KV head) of a decode step: quantize the
    new K/V token into the oracle's own cache of that group, then decode all
    the group's query heads over the context.  Cache prefill is untimed."""
    import numpy as np

    from online_kv_cache_tq_gb300 import workloads as W
    from oracle import attention, engine
    name, seed, ctx, kvh = task
    cfg = W.CONFIGS[name]
    book = engine.build(k_bits=cfg["k_bits"], v_bits=cfg["v_bits"], qjl_m=cfg["qjl_m"], seed=cfg["seed"])
    rng = np.random.default_rng(seed)
    prof = (cfg.get("log_uniform"), cfg.get("outliers", 0), cfg.get("outlier_scale", 1.0))
    ks = W.channel_scales(seed, cfg["n_kv"], *prof)[kvh]
    vs = W.channel_scales(seed + 1, cfg["n_kv"], *prof)[kvh]
    bs = cfg["block_size"]
    nblk = (ctx + bs - 1) // bs
    k = W.bf16_round_numpy(rng.standard_normal((ctx, 1, 128)) * ks)
    v = W.bf16_round_numpy(rng.standard_normal((ctx, 1, 128)) * vs)
    cache = engine.empty_cache(book, nblk, 1, bs)
    engine.append(cache, book, k[:-1], v[:-1], np.arange(ctx - 1))
    group = cfg["n_q"] // cfg["n_kv"]
    q = W.bf16_round_numpy(rng.standard_normal((group, 128)))
    table = np.arange(nblk)
    t0 = time.perf_counter()
    engine.append(cache, book, k[-1:], v[-1:], np.array([ctx - 1]))
    for h in range(group):
        attention.decode_attention(q[h], cache, table, ctx, 0, book)
    return time.perf_counter() - t0


def _pool_init():
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"


def oracle_throughput(name, n_groups, seed, pool, processes):
    """Decode tokens/s of the oracle on ``processes`` host cores, measured on
    ``n_groups`` sampled (sequence, KV head) groups of the workload."""
    import numpy as np

    from online_kv_cache_tq_gb300 import workloads as W
    cfg = W.CONFIGS[name]
    ctx = W.context_lengths(cfg, seed)
    rng = np.random.default_rng(seed + 99)
    tasks = [(name, seed + i, int(ctx[rng.integers(len(ctx))]), int(rng.integers(cfg["n_kv"])))
             for i in range(n_groups)]
    times = pool.map(_oracle_group, tasks)
    per_group = float(np.mean(times)) * float(np.mean(ctx)) / float(np.mean([t[2] for t in tasks]))
    return processes / (cfg["n_kv"] * per_group), n_groups


def oracle_pool():
    _pool_init()
    procs = max(1, min(16, os.cpu_count() or 1))
    return mp.get_context("spawn").Pool(procs, initializer=_pool_init), procs


def workload_config(name, cfg, copies):
    ctx = cfg["context"]
    out = {"workload": name, "batch": cfg["batch"], "n_q_heads": cfg["n_q"], "n_kv_heads": cfg["n_kv"],
           "head_dim": 128, "context": list(ctx) if isinstance(ctx, tuple) else ctx,
           "k_bits": cfg["k_bits"], "v_bits": cfg["v_bits"], "qjl_m": cfg["qjl_m"],
           "block_size": cfg["block_size"], "input_dtype": cfg["dtype"], "parallelism": "replicas"}
    if copies is not None:
        out["l2"] = ("inputs larger than L2: steps rotate over %d cache copies" % copies if copies > 1
                     else "inputs larger than L2: one cache larger than 2x L2")
    return out


def run_reference(args):
    rank, world, _ = rank_env()
    if rank != 0:
        return 0
    from online_kv_cache_tq_gb300 import workloads as W
    cfg = W.CONFIGS[args.workload]
    pool, procs = oracle_pool()
    groups = max(procs, 8)
    for i in range(args.warmup):
        oracle_throughput(args.workload, groups, 1 + i, pool, procs)
    vals = []
    t0 = time.perf_counter()
    for i in range(args.steps):
        vals.append(oracle_throughput(args.workload, groups, 100 + i, pool, procs)[0])
    wall = time.perf_counter() - t0
    pool.close()
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * wall / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, cfg, None),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": procs, "kind": "oracle",
                         "sample": "%d (sequence, KV head) groups per step, each: quantize the new token + decode "
                                   "%d query heads over its context; scaled to the full batch" %
                                   (groups, cfg["n_q"] // cfg["n_kv"])},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    rank, world, local_rank = rank_env()
    pool = procs = None
    if rank == 0 and not args.no_cpu_baseline:
        pool, procs = oracle_pool()         # spawned before any GPU work
    init_ranks("nccl" if world > 1 else "gloo")
    wl, max_ms, attn_ms, clock_info, e2e, quant = run_ours(args, rank, world, local_rank)
    if rank != 0:
        return 0
    ms_per_step = max_ms / args.steps
    peak, peak_src = hbm_peak()
    achieved = wl.cache_bytes / (attn_ms * 1e-3) / 1e9
    tc = wl.B.tq_decode_kernel_kind(wl.book, wl.n_q, wl.n_kv)
    kernel = ("attention_tc_kernel<%d>" if tc else "attention_kernel<%d>") % (wl.n_q // wl.n_kv)
    line = {
        "metric": METRIC, "value": world * wl.batch / (ms_per_step * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(args.workload, wl.cfg, len(wl.caches)),
        "hbm_gbs_step": wl.cache_bytes / (ms_per_step * 1e-3) / 1e9,
        "kv_token_heads_per_s": world * float(wl.ctx.sum()) * wl.n_kv / (ms_per_step * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": recorded_traffic(kernel, args.workload), "kernel": kernel,
                     "peak_source": peak_src + " hbm_gbs", "algorithmic_bytes_per_launch": wl.cache_bytes,
                     "launch_ms": attn_ms},
        "gpu_launches": wl.launches_per_step * args.steps,
        "clocks": clock_info,
        "e2e": e2e,
        "prefill_quantize": quant,
    }
    if pool is not None:
        value, groups = oracle_throughput(args.workload, args.cpu_groups, 7, pool, procs)
        pool.close()
        line["cpu_baseline"] = {"value": value, "unit": "tokens/s", "cores": procs, "kind": "oracle",
                                "sample": "%d sampled (sequence, KV head) groups: quantize the new token + decode "
                                          "the group's query heads over its context, scaled to the batch" % groups}
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
