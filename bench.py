#!/usr/bin/env python3
"""Benchmark of the TurboQuant KV-cache hot path on GB300.

One step = the whole per-layer decode path for one batch: quantize-append of
each sequence's new K/V token into the packed cache, then decode attention of
every query head over the full packed context (query preparation, split-K
attention with the merge and back-rotation in the same kernel).

Headline workload (the largest single-GPU configuration): a Llama-3-70B-shaped
paged decode layer -- batch 64, 64 query heads, 8 KV heads, d 128, context
lengths drawn uniformly from [1024, 32768], 64-token blocks under a shuffled
block table, 3-bit K (2-bit MSE + 1-bit QJL) and 3-bit V, synthetic bf16 K/V
with log-uniform per-channel scales.  The same JSON line carries secondary
figures for the other workloads: the Llama-3-8B decode layer, the 128 K-token
long-context case, the fp32 single-head case and the prefill quantize-append
at 2, 3 and 4 bits.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on the host cores on the headline workload (bounded sample per step).
Multi-GPU: one process per GPU under torchrun; every rank runs its own
replica (different seeds: weak scaling, no data-path collective); the step
time is the max over ranks.  The oracle runs only in the CPU leg: the timed
oracle sample (cpu_baseline) and, on the same host pass, the parity figures
(the GPU's codes and outputs against the oracle on sampled inputs).
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
METRIC = "decode attn tokens/s & HBM GB/s (% of peak) over 3-bit KV; quantize vectors/s"
HEADLINE = "c5_llama3_70b_paged"
SECONDARY_DECODE = ("c2_llama3_8b_decode", "c4_long_context", "c5_llama3_70b_paged_fp16_norms",
                    "c2_llama3_8b_decode_polar")
CODE_EXEMPT = 1e-5          # codes within this distance of a boundary (unit-vector units) may differ
ATTN_TOL = 1e-3             # max |o_gpu - o_oracle| / max_t ||v_hat_t||


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=HEADLINE)
    p.add_argument("--cpu-groups", type=int, default=32, help="oracle (sequence, KV head) groups timed")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle leg (timing and parity)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-secondary", action="store_true", help="headline workload only")
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

def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh)
    except (OSError, ValueError):
        return None


def hbm_peak():
    p = _peaks()
    try:
        return float(p["hbm_gbs"]), "measured"
    except (TypeError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Burst bf16 dense tensor TFLOP/s (a kernel timed alone), measured or fallback."""
    p = _peaks()
    try:
        return float(p["bf16_tflops"]), "measured"
    except (TypeError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


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


def events(n):
    import torch
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]


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
        self.seed = seed
        self.batch, self.n_q, self.n_kv = cfg["batch"], cfg["n_q"], cfg["n_kv"]
        self.book = B.Codebook(k_bits=cfg["k_bits"], v_bits=cfg["v_bits"], qjl_m=cfg["qjl_m"], seed=cfg["seed"],
                               block_size=cfg["block_size"], device=device, norm_bits=cfg.get("norm_bits", 32),
                               codec=cfg.get("codec", 0))
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
        # quantize K, quantize V, prepare), then the partials kernel, which merges in place or
        # is followed by a merge launch
        self.plan = B.tq_decode_plan(self.book, self.batch, self.n_q, self.n_kv, self.max_ctx)
        self.tc = self.plan["tensor_cores"] == 1
        # (a PolarQuant step appends keys and values in two launches before the preparation)
        prep = 3 if self.book.codec == 1 or self.batch * self.n_kv > 1024 else 1
        self.launches_per_step = prep + (1 if self.plan["merge_in_partials"] else 2)

    def step(self, i):
        """One decode step: tq_decode_step (append the new K/V token of every
        sequence, then decode attention), inputs resident on the device."""
        self.B.tq_decode_step(self.book, self.k_new, self.v_new, self.dtype_code, self.q, self.dtype_code,
                              self.batch, self.n_q, self.n_kv, self.views[i % len(self.views)], self.table_d,
                              self.max_blocks, self.ctx_d, self.max_ctx, 0.0, self.out, self.ws, self.ws_bytes)

    def staged_step(self, i, ev):
        """The same step through the staged calls: the append + query
        preparation, then (between the events) the partials kernel exactly as
        the step runs it (merging in place when the step's plan says so),
        then the merge launch when the plan has one."""
        B = self.B
        view = self.views[i % len(self.views)]
        B.tq_decode_step_prepare(self.book, self.k_new, self.v_new, self.dtype_code, self.q, self.dtype_code,
                                 self.batch, self.n_q, self.n_kv, view, self.table_d, self.max_blocks, self.ctx_d,
                                 self.max_ctx, self.ws, self.ws_bytes)
        fused = self.plan["merge_in_partials"] == 1
        ev[0].record()
        B.tq_decode_partials(self.book, self.batch, self.n_q, self.n_kv, view, self.table_d, self.max_blocks,
                             self.ctx_d, self.max_ctx, 0.0, self.ws, self.ws_bytes, out=self.out if fused else None)
        ev[1].record()
        if not fused:
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

    def kernel_name(self):
        if self.book.codec == 1:
            return "polar_attention_kernel<%d>" % (self.n_q // self.n_kv)
        return ("attention_tc_kernel<%d>" if self.tc else "attention_kernel<%d>") % (self.n_q // self.n_kv)

    def parity_sample(self, n_groups, seed):
        """Host copies for the oracle check of ``n_groups`` sampled (sequence,
        KV head) groups: each group's sequence blocks of every cache field (the
        state the last step decoded), the group's queries and GPU outputs."""
        np, torch = self.np, self.torch
        rng = np.random.default_rng(seed)
        groups = sorted({(int(rng.integers(self.batch)), int(rng.integers(self.n_kv))) for _ in range(n_groups)})
        out_h = self.out.cpu().numpy()
        q_h = self.q.double().cpu().numpy()
        bs = self.cfg["block_size"]
        items = []
        for b, kvh in groups:
            n_blk = (int(self.ctx[b]) + bs - 1) // bs
            idx = torch.as_tensor(self.table[b, :n_blk].astype(np.int64), device="cuda")
            fields = {name: t.index_select(0, idx).cpu().numpy() for name, t in self.caches[0].items()}
            g = self.n_q // self.n_kv
            items.append({"b": b, "kvh": kvh, "ctx": int(self.ctx[b]), "cache": fields,
                          "q": q_h[b, kvh * g:(kvh + 1) * g], "out": out_h[b, kvh * g:(kvh + 1) * g]})
        return {"workload": self.name, "k_bits": self.cfg["k_bits"], "v_bits": self.cfg["v_bits"],
                "qjl_m": self.cfg["qjl_m"], "seed": self.cfg["seed"], "codec": self.book.codec, "groups": items}


def measure_decode(name, steps, warmup, seed, clocks=None, with_e2e=False, parity_groups=0):
    """Decode step time and the partials kernel's time for one workload."""
    import torch
    wl = DecodeWorkload(name, torch.cuda.current_device(), seed)
    for i in range(warmup):
        wl.step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clocks is not None:
        clocks.start()
    barrier()
    torch.cuda.synchronize()
    start.record()
    for i in range(steps):
        wl.step(warmup + i)
    end.record()
    torch.cuda.synchronize()
    barrier()
    # the dominant kernel's duration: the same steps through the staged calls,
    # with events around each partials launch on the launching stream
    ev = events(steps)
    for i in range(steps):
        wl.staged_step(warmup + steps + i, ev[i])
    torch.cuda.synchronize()
    clock_info = clocks.stop() if clocks is not None else None
    if wl.B.tq_get_last_device_error(wl.book):
        raise RuntimeError("device error during the %s benchmark" % name)
    # one more step, so that the output and cache match for the parity sample
    wl.step(0)
    torch.cuda.synchronize()
    step_ms = start.elapsed_time(end) / steps
    part_ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    res = {"wl": wl, "step_ms": step_ms, "partials_ms": part_ms, "clocks": clock_info}
    if with_e2e:
        res["e2e"] = wl.e2e(steps, min(warmup, 5))
    if parity_groups:
        res["parity_sample"] = wl.parity_sample(parity_groups, seed + 5)
    return res


def decode_summary(res, world, dev):
    """Secondary-line figures of one decode workload (max over ranks)."""
    wl = res["wl"]
    step_ms = max_over_ranks(res["step_ms"], dev)
    part_ms = max_over_ranks(res["partials_ms"], dev)
    peak, src = hbm_peak()
    achieved = wl.cache_bytes / (part_ms * 1e-3) / 1e9
    return {
        "workload": wl.name, "ms_per_step": step_ms, "tokens_per_s": world * wl.batch / (step_ms * 1e-3),
        "kv_token_heads_per_s": world * float(wl.ctx.sum()) * wl.n_kv / (step_ms * 1e-3),
        "hbm_gbs_step": wl.cache_bytes / (step_ms * 1e-3) / 1e9,
        "bytes_per_token_head": wl.bytes_per_token_head,
        "compression_vs_bf16": 4.0 * 128 / wl.bytes_per_token_head,
        "plan": wl.plan,
        "partials": {"kernel": wl.kernel_name(), "launch_ms": part_ms, "achieved_gbs": achieved,
                     "frac": achieved / peak, "peak_source": src + " hbm_gbs",
                     "algorithmic_bytes_per_launch": wl.cache_bytes,
                     "traffic": recorded_traffic(wl.kernel_name(), wl.name)},
        "context_tokens": int(wl.ctx.sum()), "l2": l2_note(len(wl.caches)),
        "norm_bits": wl.book.norm_bits,
    }


def l2_note(copies):
    return ("inputs larger than L2: steps rotate over %d cache copies" % copies if copies > 1
            else "inputs larger than L2: one cache larger than 2x L2")


# ------------------------------------------------------ quantize (ours) --

def measure_quantize(bits, steps, warmup, sample_tokens=0, polar=False):
    """Prefill quantize-append of 32768 tokens x 8 KV heads (bf16, Student-t
    outlier channels) at ``bits`` per K (bits - 1 MSE + QJL) and V, or with
    the PolarQuant codec (polar: bits unused, no parity sample); two input
    copies rotated so the 128 MB of inputs are read from HBM."""
    import numpy as np
    import torch

    from online_kv_cache_tq_gb300 import binding as B
    from online_kv_cache_tq_gb300 import cache as C
    from online_kv_cache_tq_gb300 import workloads as W
    cfg = W.CONFIGS["c3_prefill_quantize"]
    n_tok, n_kv = cfg["tokens"], cfg["n_kv"]
    if polar:
        book = B.Codebook(k_bits=0, v_bits=0, qjl_m=0, seed=cfg["seed"], block_size=cfg["block_size"],
                          device=torch.cuda.current_device(), codec=B.TQ_CODEC_POLAR)
    else:
        book = B.Codebook(k_bits=bits, v_bits=bits, qjl_m=cfg["qjl_m"], seed=cfg["seed"],
                          block_size=cfg["block_size"], device=torch.cuda.current_device())
    g = torch.Generator(device="cuda")
    g.manual_seed(cfg["seed"] + bits)
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
    ev = events(steps)
    torch.cuda.synchronize()
    for i in range(steps):
        ev[i][0].record()
        append(i)
        ev[i][1].record()
    torch.cuda.synchronize()
    if B.tq_get_last_device_error(book):
        raise RuntimeError("device error during the quantize measurement")
    secs = sum(a.elapsed_time(b) for a, b in ev) * 1e-3 / steps
    vectors = 2 * n_tok * n_kv
    field = C.cache_bytes_per_token_head(book)
    nbytes = vectors * 256 + n_tok * n_kv * field            # bf16 reads + packed writes
    flops = n_tok * n_kv * (2 * 32768) + n_tok * n_kv * 32768  # K: rotation + QJL, V: rotation
    hbm, _ = hbm_peak()
    tensor, tensor_src = bf16_peak()
    if polar:
        res = {"workload": "c3_prefill_quantize", "codec": "polar", "tokens": n_tok, "n_kv_heads": n_kv,
               "ms_per_append": secs * 1e3, "vectors_per_s": vectors / secs,
               "hbm_gbs": nbytes / secs / 1e9, "hbm_frac": nbytes / secs / 1e9 / hbm,
               "algorithmic_bytes_per_append": nbytes,
               "note": "PolarQuant records (64 B + float32 radius per vector); the rotation and the polar "
                       "levels run on the CUDA cores"}
        return res, None
    kb = bits - 1
    rec = [recorded_traffic(k, "c3_prefill_quantize") for k in
           ("quantize_tc_kernel<%d,1,0>" % kb, "quantize_tc_kernel<%d,0,1>" % bits)]
    traffic = sum(rec) if all(r is not None for r in rec) else None
    res = {"workload": "c3_prefill_quantize", "tokens": n_tok, "n_kv_heads": n_kv, "k_bits": bits, "v_bits": bits,
           "ms_per_append": secs * 1e3, "vectors_per_s": vectors / secs,
           "hbm_gbs": nbytes / secs / 1e9, "hbm_frac": nbytes / secs / 1e9 / hbm,
           "algorithmic_tflops": flops / secs / 1e12, "tensor_frac": flops / secs / 1e12 / tensor,
           "tensor_peak_source": tensor_src + " bf16_tflops",
           "algorithmic_bytes_per_append": nbytes, "traffic_bytes_per_append": traffic,
           "note": "algorithmic flops; the bf16 hi/lo splitting runs 2 (rotation) and 3 (QJL) tensor passes"}
    sample = None
    if sample_tokens:
        # the last append wrote inputs[(steps - 1) % 2]: sampled tokens and their cache rows on the host
        k, v = inputs[(steps - 1) % 2]
        toks = np.sort(np.random.default_rng(bits).choice(n_tok, size=sample_tokens, replace=False))
        idx = torch.as_tensor(toks, device="cuda")
        sample = {"bits": bits, "qjl_m": cfg["qjl_m"], "seed": cfg["seed"], "block_size": cfg["block_size"],
                  "slots": toks, "k": k.index_select(0, idx).double().cpu().numpy(),
                  "v": v.index_select(0, idx).double().cpu().numpy(),
                  "cache": {name: t.cpu().numpy() for name, t in cache.items()}}
    return res, sample


def measure_single_head_fp32(steps, warmup):
    """The fp32 single-head workload: quantize-append of 4096 keys and 4096
    values (4 outlier channels x20) and decode of one query over them."""
    import numpy as np
    import torch

    from online_kv_cache_tq_gb300 import binding as B
    from online_kv_cache_tq_gb300 import cache as C
    from online_kv_cache_tq_gb300 import workloads as W
    cfg = W.CONFIGS["c1_single_head_parity"]
    n = cfg["context"]
    book = B.Codebook(k_bits=cfg["k_bits"], v_bits=cfg["v_bits"], qjl_m=cfg["qjl_m"], seed=cfg["seed"],
                      block_size=cfg["block_size"], device=torch.cuda.current_device())
    g = torch.Generator(device="cuda")
    g.manual_seed(cfg["seed"])
    k = W.gaussian_tokens(n, W.channel_scales(0, 1, None, 4, 20.0), torch.float32, "cuda", g)
    v = W.gaussian_tokens(n, W.channel_scales(1, 1, None, 4, 20.0), torch.float32, "cuda", g)
    cache = C.allocate_cache(book, n // cfg["block_size"], 1)
    view = C.cache_view(book, cache)
    slots = torch.arange(n, device="cuda", dtype=torch.int64)
    q = W.queries(1, 1, torch.float32, "cuda", g)
    ctx = torch.full((1,), n, dtype=torch.int32, device="cuda")
    ws, nbytes = C.allocate_workspace(book, 1, 1, n)
    out = torch.empty((1, 1, 128), device="cuda")
    for _ in range(warmup):
        B.tq_quantize_append(book, k, v, B.TQ_FP32, n, 1, slots, view)
        B.tq_decode_attention(book, q, B.TQ_FP32, 1, 1, 1, view, None, n // cfg["block_size"], ctx, n, 0.0, out,
                              ws, nbytes)
    eq, ed = events(steps), events(steps)
    torch.cuda.synchronize()
    for i in range(steps):
        eq[i][0].record()
        B.tq_quantize_append(book, k, v, B.TQ_FP32, n, 1, slots, view)
        eq[i][1].record()
        ed[i][0].record()
        B.tq_decode_attention(book, q, B.TQ_FP32, 1, 1, 1, view, None, n // cfg["block_size"], ctx, n, 0.0, out,
                              ws, nbytes)
        ed[i][1].record()
    torch.cuda.synchronize()
    if B.tq_get_last_device_error(book):
        raise RuntimeError("device error during the fp32 single-head measurement")
    tq_ms = sum(a.elapsed_time(b) for a, b in eq) / steps
    td_ms = sum(a.elapsed_time(b) for a, b in ed) / steps
    return {"workload": "c1_single_head_parity", "input_dtype": "fp32", "vectors": 2 * n,
            "quantize_ms": tq_ms, "quantize_vectors_per_s": 2 * n / (tq_ms * 1e-3),
            "decode_ms": td_ms, "decode_tokens_per_s": 1.0 / (td_ms * 1e-3),
            "decode_kv_token_heads_per_s": n / (td_ms * 1e-3),
            "note": "latency-bound sizes: one head, 4096 tokens"}


BIAS_CASES = ((1, 0), (2, 128), (2, 0), (3, 128))   # (key bits, QJL rows): MSE-only and with the QJL bit


def bias_sample(n=4096, n_queries=16, seed=5):
    """Keys ~ N(0, I) (bf16) quantized by the GPU for each of BIAS_CASES, with
    host copies of the inputs and of the cache rows the GPU wrote, and
    queries ~ N(0, I): the material of the inner-product bias figures."""
    import numpy as np
    import torch

    from online_kv_cache_tq_gb300 import binding as B
    from online_kv_cache_tq_gb300 import cache as C
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    k = torch.randn((n, 1, 128), generator=g, device="cuda").to(torch.bfloat16)
    slots = torch.arange(n, device="cuda", dtype=torch.int64)
    cases = []
    for k_bits, qjl in BIAS_CASES:
        book = B.Codebook(k_bits=k_bits, v_bits=2, qjl_m=qjl, seed=0, block_size=64,
                          device=torch.cuda.current_device())
        cache = C.allocate_cache(book, n // 64, 1)
        B.tq_quantize_append(book, k, None, B.TQ_BF16, n, 1, slots, C.cache_view(book, cache))
        torch.cuda.synchronize()
        cases.append({"k_bits": k_bits, "qjl_m": qjl,
                      "cache": {f: t.cpu().numpy() for f, t in cache.items() if f.startswith("k_")}})
    q = np.random.default_rng(seed).standard_normal((n_queries, 128))
    return {"x": k.double().cpu().numpy().reshape(n, 128), "q": q, "cases": cases}


def _bias_figures(sample):
    """Slope of the estimated inner products on the true ones, sum e t / sum t^2
    over (key, query) pairs, for keys decoded from the GPU's codes: stage 1
    alone shrinks inner products by E||c||^2 = 1 - D_mse (d c_1^2, near 2/pi,
    at 1 bit; 甲子光年 article §2 第二階段), the QJL bit removes the shrinkage.
    The standard error treats keys as independent."""
    import numpy as np

    from oracle import attention, codebook, engine, packing, quantize
    x, q = sample["x"], sample["q"]
    true = x @ q.T
    out = []
    for case in sample["cases"]:
        ref = engine.build(k_bits=case["k_bits"], v_bits=2, qjl_m=case["qjl_m"], seed=0)
        c = case["cache"]
        rows = c["k_codes"].reshape(-1, c["k_codes"].shape[-1])[:len(x)]
        codes = packing.unpack_planes(rows, ref["k_bits"], 128)
        xhat = quantize.reconstruct_mse(c["k_norm"].reshape(-1)[:len(x)], codes, ref["rot"], ref["k_levels"])
        est = xhat @ q.T
        if case["qjl_m"]:
            signs = packing.unpack_signs(c["k_qjl"].reshape(-1, 16)[:len(x)], ref["proj"].shape[0])
            gamma = c["k_rnorm"].reshape(-1)[:len(x)]
            est = est + np.stack([attention.qjl_estimate(qq, gamma, signs, ref["proj"]) for qq in q], axis=1)
        s_i, w_i = np.sum(est * true, axis=1), np.sum(true * true, axis=1)
        slope = float(s_i.sum() / w_i.sum())
        stderr = float(np.sqrt(np.sum((s_i - slope * w_i) ** 2)) / w_i.sum())
        expect = 1.0 if case["qjl_m"] else 1.0 - codebook.mse_distortion(128, ref["k_levels"], ref["k_bounds"])
        out.append({"k_bits": case["k_bits"], "qjl_m": case["qjl_m"], "mse_bits": ref["k_bits"],
                    "slope": slope, "stderr": stderr, "expected": float(expect)})
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    torch.cuda.set_device(local_rank)
    import __graft_entry__
    __graft_entry__.build()
    dev = "cuda" if world > 1 else "cpu"
    want_parity = rank == 0 and not args.no_cpu_baseline
    head = measure_decode(args.workload, args.steps, args.warmup, rank_seed(0, rank), ClockSampler(local_rank),
                          with_e2e=not args.no_e2e, parity_groups=6 if want_parity else 0)
    out = {"head": head, "secondary": {}, "quant_samples": [], "decode_samples": []}
    if want_parity:
        out["decode_samples"].append(head.pop("parity_sample"))
    if not args.no_secondary:
        steps = max(20, min(args.steps, 100))
        for name in SECONDARY_DECODE:
            if name == args.workload:
                continue
            res = measure_decode(name, steps, args.warmup, rank_seed(0, rank), parity_groups=4 if want_parity else 0)
            out["secondary"][name] = decode_summary(res, world, dev)
            if want_parity:
                out["decode_samples"].append(res.pop("parity_sample"))
            del res
        for bits in (2, 3, 4):
            res, sample = measure_quantize(bits, 20, 3, sample_tokens=256 if want_parity else 0)
            out["secondary"]["c3_prefill_quantize_b%d" % bits] = res
            if sample is not None:
                out["quant_samples"].append(sample)
        out["secondary"]["c3_prefill_quantize_polar"] = measure_quantize(0, 20, 3, polar=True)[0]
        out["secondary"]["c1_single_head_parity"] = measure_single_head_fp32(20, 3)
    if want_parity:
        out["bias_sample"] = bias_sample()
    return out


# ----------------------------------------------------- oracle (CPU leg) --

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
    ``n_groups`` sampled (sequence, KV head) groups of the workload: the mean
    group time, scaled to the batch's mean context, times the groups of a step."""
    import numpy as np

    from online_kv_cache_tq_gb300 import workloads as W
    cfg = W.CONFIGS[name]
    ctx = W.context_lengths(cfg, seed)
    rng = np.random.default_rng(seed + 99)
    tasks = [(name, seed + i, int(ctx[rng.integers(len(ctx))]), int(rng.integers(cfg["n_kv"])))
             for i in range(n_groups)]
    times = pool.map(_oracle_group, tasks)
    per_group = float(np.mean(times)) * float(np.mean(ctx)) / float(np.mean([t[2] for t in tasks]))
    step_s = cfg["batch"] * cfg["n_kv"] * per_group / processes
    return cfg["batch"] / step_s, n_groups


def oracle_pool():
    _pool_init()
    procs = max(1, min(16, os.cpu_count() or 1))
    return mp.get_context("spawn").Pool(procs, initializer=_pool_init), procs


def _decode_parity_group(task):
    """Worst normalised attention error of one sampled group's G heads: the
    oracle decodes the GPU's own packed cache (identical codes)."""
    import numpy as np

    from oracle import attention, engine
    cfg, item = task
    if cfg.get("codec", 0) == 1:
        book = engine.build(codec="polar", seed=cfg["seed"])
    else:
        book = engine.build(k_bits=cfg["k_bits"], v_bits=cfg["v_bits"], qjl_m=cfg["qjl_m"], seed=cfg["seed"])
    table = np.arange(item["cache"]["k_norm"].shape[0])
    worst = 0.0
    for h in range(item["q"].shape[0]):
        expect, vmax = attention.decode_attention(item["q"][h], item["cache"], table, item["ctx"], item["kvh"],
                                                  book)
        worst = max(worst, float(np.max(np.abs(item["out"][h] - expect)) / vmax))
    return worst


def _quant_parity(sample):
    """Exempt and non-exempt code / sign disagreements of sampled vectors (the
    GPU's cache rows against the oracle's encoding of the same inputs)."""
    import numpy as np

    from oracle import engine, packing, quantize
    bits = sample["bits"]
    ref = engine.build(k_bits=bits, v_bits=bits, qjl_m=sample["qjl_m"], seed=sample["seed"])
    cache, slots, bs = sample["cache"], sample["slots"], sample["block_size"]
    n_kv = cache["k_norm"].shape[1]
    rep = {"bits": bits, "vectors": 0, "exempt_codes": 0, "near_boundary": 0, "non_exempt_codes": 0,
           "exempt_signs": 0, "non_exempt_signs": 0}
    for which in ("k", "v"):
        x = sample[which].reshape(-1, 128)
        rows = np.stack([packing.slot_index(slots, h, n_kv, bs) for h in range(n_kv)], axis=1).reshape(-1)
        if which == "k":
            flat = cache["k_codes"].reshape(-1, cache["k_codes"].shape[-1])
            got = packing.unpack_planes(flat[rows], ref["k_bits"], 128)
        else:
            got = np.stack([packing.read_value_codes(cache["v_codes"], slots, h) for h in range(n_kv)], axis=1)
            got = got.reshape(-1, 128)
        norm = cache[which + "_norm"].reshape(-1)[rows]
        bounds = ref[which + "_bounds"]
        _, y, codes = quantize.encode_mse(x, ref["rot"], bounds)
        diff = got != codes
        exempt = quantize.boundary_distance(y, bounds) < CODE_EXEMPT
        rep["vectors"] += len(x)
        rep["exempt_codes"] += int((diff & exempt).sum())
        rep["near_boundary"] += int(exempt.sum())
        rep["non_exempt_codes"] += int((diff & ~exempt).sum())
        if which == "k" and ref["qjl_m"]:
            _, signs, z = quantize.encode_qjl(x, norm, got, ref["rot"], ref["k_levels"], ref["proj"])
            flat = cache["k_qjl"].reshape(-1, cache["k_qjl"].shape[-1])
            gs = packing.unpack_signs(flat[rows], ref["proj"].shape[0])
            xn = np.linalg.norm(x, axis=1)
            ex = np.abs(z) < CODE_EXEMPT * xn[:, None] * np.linalg.norm(ref["proj"], axis=1)[None, :]
            d = gs != signs
            rep["exempt_signs"] += int((d & ex).sum())
            rep["non_exempt_signs"] += int((d & ~ex).sum())
    return rep


def cpu_leg(name, n_groups, pool, procs, decode_samples, quant_samples, bias=None):
    """The oracle on the host cores: its timed decode throughput on a bounded
    sample of the workload (cpu_baseline), then the parity figures of the GPU
    outputs and codes sampled by the GPU runs."""
    value, groups = oracle_throughput(name, n_groups, 7, pool, procs)
    base = {"value": value, "unit": "tokens/s", "cores": procs, "kind": "oracle",
            "sample": "%d sampled (sequence, KV head) groups: quantize the new token + decode the group's "
                      "query heads over its context, scaled to the batch" % groups}
    parity = {"attention_tolerance": ATTN_TOL, "code_exempt_band": CODE_EXEMPT, "decode": {}, "quantize": {}}
    for s in decode_samples:
        cfg = {k: s[k] for k in ("k_bits", "v_bits", "qjl_m", "seed", "codec")}
        worst = pool.map(_decode_parity_group, [(cfg, it) for it in s["groups"]])
        parity["decode"][s["workload"]] = {
            "groups": len(worst), "heads": int(sum(it["q"].shape[0] for it in s["groups"])),
            "worst_normalised_error": max(worst), "within_tolerance": max(worst) <= ATTN_TOL}
    for rep in pool.map(_quant_parity, quant_samples):
        parity["quantize"]["c3_prefill_quantize_b%d" % rep["bits"]] = rep
    if bias is not None:
        parity["inner_product_bias"] = _bias_figures(bias)
    return base, parity


def workload_config(name, cfg, copies):
    ctx = cfg["context"]
    out = {"workload": name, "batch": cfg["batch"], "n_q_heads": cfg["n_q"], "n_kv_heads": cfg["n_kv"],
           "head_dim": 128, "context": list(ctx) if isinstance(ctx, tuple) else ctx,
           "k_bits": cfg["k_bits"], "v_bits": cfg["v_bits"], "qjl_m": cfg["qjl_m"],
           "block_size": cfg["block_size"], "input_dtype": cfg["dtype"],
           "shuffled_block_table": bool(cfg.get("shuffled_table", False)), "parallelism": "replicas"}
    if copies is not None:
        out["l2"] = l2_note(copies)
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
        "config": workload_config(args.workload, cfg, 1),
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
    res = run_ours(args, rank, world, local_rank)
    head = res["head"]
    wl = head["wl"]
    dev = "cuda" if world > 1 else "cpu"
    step_ms = max_over_ranks(head["step_ms"], dev)
    part_ms = max_over_ranks(head["partials_ms"], dev)
    e2e = None
    if "e2e" in head:
        secs, h2d, d2h = head["e2e"]
        secs = max_over_ranks(secs, dev)
        e2e = {"value": world * wl.batch * args.steps / secs, "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    if rank != 0:
        return 0
    peak, peak_src = hbm_peak()
    achieved = wl.cache_bytes / (part_ms * 1e-3) / 1e9
    kernel = wl.kernel_name()
    line = {
        "metric": METRIC, "value": world * wl.batch / (step_ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(args.workload, wl.cfg, len(wl.caches)),
        "hbm_gbs_step": wl.cache_bytes / (step_ms * 1e-3) / 1e9,
        "kv_token_heads_per_s": world * float(wl.ctx.sum()) * wl.n_kv / (step_ms * 1e-3),
        "bytes_per_token_head": wl.bytes_per_token_head,
        "compression_vs_bf16": 4.0 * 128 / wl.bytes_per_token_head,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": recorded_traffic(kernel, args.workload), "kernel": kernel,
                     "peak_source": peak_src + " hbm_gbs", "algorithmic_bytes_per_launch": wl.cache_bytes,
                     "launch_ms": part_ms},
        "gpu_launches": wl.launches_per_step * args.steps,
        "plan": wl.plan,
        "clocks": head["clocks"],
        "e2e": e2e,
        "secondary": res["secondary"],
    }
    if pool is not None:
        base, parity = cpu_leg(args.workload, args.cpu_groups, pool, procs, res["decode_samples"],
                               res["quant_samples"], res.get("bias_sample"))
        pool.close()
        line["cpu_baseline"] = base
        line["parity"] = parity
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
