"""Shared helpers of the GPU parity tests: run the library through the C ABI
and compare with the oracle under the acceptance rules.

Acceptance (as the method's tolerances are stated for this engine):
* codes bit-exact except coordinates whose unit rotated value lies within
  1e-5 of a decision boundary (distance in units of ||x||); the count of such
  exempt disagreements is reported;
* QJL sign bits bit-exact except where |(S r)_k| < 1e-5 ||x|| ||S_k||; the
  oracle recomputes the residual from the GPU's codes and stored norm;
* attention outputs computed from identical codes (the GPU's packed cache is
  read back and decoded by the oracle) agree to
  max_abs(o_gpu - o_oracle) / max_t ||v_hat_t|| <= 1e-3 per (sequence, head).
"""
import numpy as np
import torch

from online_kv_cache_tq_gb300 import binding as B
from online_kv_cache_tq_gb300 import cache as C
from online_kv_cache_tq_gb300 import workloads as W
from oracle import attention, engine, packing, quantize

CODE_EXEMPT = 1e-5
ATTN_TOL = 1e-3


def books(k_bits=3, v_bits=3, qjl_m=128, seed=0, block_size=64, norm_bits=32):
    gpu = B.Codebook(k_bits=k_bits, v_bits=v_bits, qjl_m=qjl_m, seed=seed, block_size=block_size, device=0,
                     norm_bits=norm_bits)
    ref = engine.build(k_bits=k_bits, v_bits=v_bits, qjl_m=qjl_m, seed=seed, norm_bits=norm_bits)
    return gpu, ref


def norm_tolerance(stored, reference):
    """|stored - reference| allowed for a norm held in ``stored``'s dtype: the
    fp32 rounding of a 128-term sum of squares (relative 2e-6), plus half an
    ulp of float16 (2^-11 relative) when the field is 16-bit."""
    rel = 2e-6 + (2.0 ** -11 if stored.dtype == np.float16 else 0.0)
    return rel * reference + 1e-30


def dtype_code(t):
    return B.TQ_BF16 if t.dtype == torch.bfloat16 else B.TQ_FP32


def generator(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return g


def quantize_into(book, cache, k, v, slots, stream=None):
    """Call tq_quantize_append for k/v [n_tok][n_kv][128] device tensors."""
    view = C.cache_view(book, cache)
    n_tok, n_kv = (k if k is not None else v).shape[:2]
    slot_t = torch.as_tensor(np.asarray(slots, dtype=np.int64), device="cuda")
    B.tq_quantize_append(book, k, v, dtype_code(k if k is not None else v), n_tok, n_kv, slot_t, view, stream)
    return slot_t


def host_cache(cache):
    torch.cuda.synchronize()
    return {name: t.cpu().numpy() for name, t in cache.items()}


def rows_at(hcache, name, slots, n_kv, block_size):
    """Rows of field ``name`` for tokens at ``slots`` (all heads): [n_tok][n_kv][...]."""
    arr = hcache[name]
    flat = arr.reshape(arr.shape[0] * arr.shape[1] * arr.shape[2], -1)
    slots = np.asarray(slots, dtype=np.int64)
    idx = np.stack([packing.slot_index(slots, h, n_kv, block_size) for h in range(n_kv)], axis=1)
    return flat[idx]


def check_mse_codes(x, got, norm_gpu, ref, which):
    """Compare GPU codes [N][d] and norms with the oracle for vectors x [N][d] (fp64)."""
    bounds = ref[which + "_bounds"]
    norm, y, codes = quantize.encode_mse(x, ref["rot"], bounds)
    diff = got != codes
    exempt = quantize.boundary_distance(y, bounds) < CODE_EXEMPT
    bad = diff & ~exempt
    assert not bad.any(), "%d non-exempt code mismatches (first at %s)" % (bad.sum(), np.argwhere(bad)[:3])
    xn = np.linalg.norm(x, axis=1)
    assert np.all(np.abs(norm_gpu.astype(np.float64) - xn) <= norm_tolerance(norm_gpu, xn))
    return int((diff & exempt).sum()), int(exempt.sum()), got


def check_qjl(x, codes_gpu, norm_gpu, packed_signs, gamma_gpu, ref):
    proj = ref["proj"]
    gamma, signs, z = quantize.encode_qjl(x, norm_gpu, codes_gpu, ref["rot"], ref["k_levels"], proj, np.float64)
    got = packing.unpack_signs(packed_signs, proj.shape[0])
    xn = np.linalg.norm(x, axis=1)
    exempt = np.abs(z) < CODE_EXEMPT * xn[:, None] * np.linalg.norm(proj, axis=1)[None, :]
    diff = got != signs
    bad = diff & ~exempt
    assert not bad.any(), "%d non-exempt QJL bit mismatches" % bad.sum()
    assert np.all(np.abs(gamma_gpu.astype(np.float64) - gamma) <= norm_tolerance(gamma_gpu, gamma) + 1e-5 * xn)
    return int((diff & exempt).sum())


def check_append(book, ref, cache, k, v, slots, sample=None):
    """Check every (or a sample of) appended (token, head) against the oracle."""
    n_kv = cache["k_norm"].shape[1]
    bs = cache["k_norm"].shape[2]
    hc = host_cache(cache)
    slots = np.asarray(slots, dtype=np.int64)
    toks = np.arange(len(slots)) if sample is None else np.asarray(sample)
    toks = toks[slots[toks] >= 0]
    report = {}
    for which, x_t in (("k", k), ("v", v)):
        if x_t is None:
            continue
        x = x_t[torch.as_tensor(toks, device=x_t.device)].double().cpu().numpy().reshape(-1, 128)
        if which == "k":
            packed = rows_at(hc, "k_codes", slots[toks], n_kv, bs).reshape(len(x), -1)
            got = packing.unpack_planes(packed, ref["k_bits"], 128)
        else:
            got = np.stack([packing.read_value_codes(hc["v_codes"], slots[toks], h) for h in range(n_kv)], axis=1)
            got = got.reshape(len(x), -1)
        norm = rows_at(hc, which + "_norm", slots[toks], n_kv, bs).reshape(-1)
        diffs, exempt, codes = check_mse_codes(x, got, norm, ref, which)
        report[which + "_exempt_code_diffs"] = diffs
        report[which + "_near_boundary"] = exempt
        if which == "k" and ref["qjl_m"]:
            signs = rows_at(hc, "k_qjl", slots[toks], n_kv, bs).reshape(len(x), -1)
            gamma = rows_at(hc, "k_rnorm", slots[toks], n_kv, bs).reshape(-1)
            report["k_exempt_sign_diffs"] = check_qjl(x, codes, norm, signs, gamma, ref)
    report["vectors"] = len(toks) * n_kv
    # exempt disagreements are rare: a coordinate lies within 1e-5 of one of
    # the 2^bits - 1 boundaries with probability ~ 2e-5 * f(t) * (2^bits - 1)
    # (f <= sqrt(d / 2 pi) ~ 4.5 for the rotated-coordinate law), below 1.5e-3
    # at 4 bits, and a code flips only within the kernel's fp32 rounding of y
    # (~1e-6, a tenth of the band): allow 1e-4 of the coordinates checked
    coords = report["vectors"] * 128
    for key in ("k_exempt_code_diffs", "v_exempt_code_diffs", "k_exempt_sign_diffs"):
        if key in report:
            assert report[key] <= 1e-4 * coords + 4, "%s = %d of %d coordinates" % (key, report[key], coords)
    return report


def decode(book, cache, q, block_table, ctx, max_context, scale=0.0, stream=None):
    batch, n_q = q.shape[:2]
    n_kv = cache["k_norm"].shape[1]
    ws, nbytes = C.allocate_workspace(book, batch, n_q, max_context)
    out = torch.full((batch, n_q, 128), float("nan"), device="cuda", dtype=torch.float32)
    view = C.cache_view(book, cache)
    table = None if block_table is None else torch.as_tensor(block_table, dtype=torch.int32, device="cuda")
    max_blocks = table.shape[1] if table is not None else cache["k_norm"].shape[0] // batch
    ctx_t = torch.as_tensor(np.asarray(ctx, dtype=np.int32), device="cuda")
    B.tq_decode_attention(book, q, dtype_code(q), batch, n_q, n_kv, view, table, max_blocks, ctx_t,
                          max_context, scale, out, ws, nbytes, stream)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def check_decode(out_gpu, hcache, q, block_table, ctx, ref, pairs, scale=None):
    """Oracle attention from the GPU's packed cache for (b, h) pairs; returns the
    worst normalised error."""
    qn = q.double().cpu().numpy()
    n_q = qn.shape[1]
    n_kv = hcache["k_norm"].shape[1]
    group = n_q // n_kv
    worst = 0.0
    for b, h in pairs:
        if int(ctx[b]) == 0:
            assert np.all(out_gpu[b, h] == 0.0)
            continue
        expect, vmax = attention.decode_attention(qn[b, h], hcache, block_table[b], int(ctx[b]), h // group,
                                                  ref, scale)
        err = np.max(np.abs(out_gpu[b, h] - expect)) / vmax
        assert err <= ATTN_TOL, "seq %d head %d: normalised error %.3g" % (b, h, err)
        worst = max(worst, err)
    return worst


def group_subset(hcache, table_row, length, kv_head, block_size):
    """The blocks of one sequence and one KV head from a host cache, as a
    one-head cache whose block table is 0, 1, ... (what the oracle reads)."""
    n_blk = (int(length) + block_size - 1) // block_size
    blocks = np.asarray(table_row[:n_blk], dtype=np.int64)
    return {name: arr[blocks][:, kv_head:kv_head + 1].copy() for name, arr in hcache.items()}


def _group_worker(task):
    qs, sub, length, book_args, scale = task
    ref = engine.build(**book_args)
    return attention.decode_attention_heads(qs, sub, np.arange(sub["k_norm"].shape[0]), length, 0, ref, scale)


def check_decode_groups(out_gpu, hcache, q, block_table, ctx, book_args, groups, scale=None, processes=1):
    """Oracle attention from the GPU's packed cache for every query head of the
    (sequence, KV head) groups listed (each group's cache decoded once), in a
    spawned process pool when processes > 1; returns the worst normalised error."""
    qn = q.double().cpu().numpy()
    n_q = qn.shape[1]
    n_kv = hcache["k_norm"].shape[1]
    bs = hcache["k_norm"].shape[2]
    g = n_q // n_kv
    tasks, keys = [], []
    for b, kvh in groups:
        heads = slice(kvh * g, (kvh + 1) * g)
        if int(ctx[b]) == 0:
            assert np.all(out_gpu[b, heads] == 0.0)
            continue
        tasks.append((qn[b, heads], group_subset(hcache, block_table[b], int(ctx[b]), kvh, bs), int(ctx[b]),
                      book_args, scale))
        keys.append((b, kvh))
    if processes > 1 and len(tasks) > 1:
        import multiprocessing as mp
        with mp.get_context("spawn").Pool(processes) as pool:
            results = pool.map(_group_worker, tasks)
    else:
        results = [_group_worker(t) for t in tasks]
    worst = 0.0
    for (b, kvh), (expect, vmax) in zip(keys, results):
        err = np.max(np.abs(out_gpu[b, kvh * g:(kvh + 1) * g] - expect)) / vmax
        assert err <= ATTN_TOL, "seq %d KV head %d: normalised error %.3g" % (b, kvh, err)
        worst = max(worst, err)
    return worst


def run_boundary_groups(ctx, n_kv, n_ctas):
    """(sequence, KV head) groups holding the first and the last item of every
    CTA run of the tensor-core decode: its items are the real 512-token chunks
    in (sequence, KV head, chunk) order, and CTA c takes the run
    [c per_cta, (c + 1) per_cta) with per_cta = ceil(items / n_ctas)."""
    chunks = (np.asarray(ctx, dtype=np.int64) + 511) // 512
    ends = np.cumsum(chunks) * n_kv                 # item index past each sequence
    starts = ends - chunks * n_kv
    total = int(ends[-1]) if len(ends) else 0
    per_cta = max(1, -(-total // n_ctas))
    picks = set()
    for c in range(n_ctas):
        for item in (c * per_cta, min(total, (c + 1) * per_cta) - 1):
            if 0 <= item < total:
                b = int(np.searchsorted(ends, item, side="right"))
                picks.add((b, int((item - starts[b]) // chunks[b])))
    return sorted(picks)


def identity_table(batch, max_blocks):
    return np.arange(batch * max_blocks, dtype=np.int32).reshape(batch, max_blocks)


def fill_cache(book, cfg, ctx, table, gen, chunk_tokens=4096):
    """Allocate a cache for ``table`` and prefill every sequence's context with
    seeded K/V of the workload's value profile."""
    n_kv = cfg["n_kv"]
    bs = cfg["block_size"]
    num_blocks = int(table.max()) + 1
    cache = C.allocate_cache(book, num_blocks, n_kv)
    dt = W.torch_dtype(cfg["dtype"])
    ks = W.channel_scales(cfg["seed"], n_kv, cfg.get("log_uniform"), cfg.get("outliers", 0),
                          cfg.get("outlier_scale", 1.0))
    vs = W.channel_scales(cfg["seed"] + 1, n_kv, cfg.get("log_uniform"), cfg.get("outliers", 0),
                          cfg.get("outlier_scale", 1.0))
    for b, length in enumerate(ctx):
        for s0 in range(0, int(length), chunk_tokens):
            n = min(chunk_tokens, int(length) - s0)
            k = W.gaussian_tokens(n, ks, dt, "cuda", gen)
            v = W.gaussian_tokens(n, vs, dt, "cuda", gen)
            quantize_into(book, cache, k, v, W.slots_for(table[b], np.arange(s0, s0 + n), bs))
    return cache


def attn_pairs(batch, n_q, count, seed):
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(batch)), int(rng.integers(n_q))) for _ in range(count)]
