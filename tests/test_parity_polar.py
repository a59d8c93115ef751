"""GPU PolarQuant codec vs the fp64 oracle, through the C ABI.

Quantize-append: every angle code bit-exact except where the pair's point
lies within 1e-5 ||x|| of the rounding boundary ray (the count is reported),
the float32 radius within the fp32 rounding of its seven levels.  Decode:
the oracle decodes the GPU's own records (identical codes), so the attention
outputs must agree to the same 1e-3 bar as the TurboQuant cache."""
import numpy as np
import pytest
import torch

from online_kv_cache_tq_gb300 import binding as B
from online_kv_cache_tq_gb300 import cache as C
from online_kv_cache_tq_gb300 import workloads as W
from oracle import engine, polar

from parity_helpers import (CODE_EXEMPT, check_decode, decode, fill_cache, generator, host_cache, quantize_into,
                            rows_at)

pytestmark = pytest.mark.gpu


def polar_books(seed=0, block_size=64):
    gpu = B.Codebook(k_bits=0, v_bits=0, qjl_m=0, seed=seed, block_size=block_size, device=0,
                     codec=B.TQ_CODEC_POLAR)
    return gpu, engine.build(codec="polar", seed=seed)


def check_records(x, records, radius_gpu, ref):
    """Codes of GPU records vs the oracle for x [N][d] (fp64); returns the
    exempt disagreements."""
    codes, radius, margins, _ = polar.encode_vectors(x, ref["rot"])
    got = polar.unpack(records)
    xn = np.linalg.norm(x, axis=1)
    exempt_diffs = 0
    for lvl, (a, b, m) in enumerate(zip(got, codes, margins), start=1):
        diff = a != b
        exempt = m < CODE_EXEMPT * xn[:, None]
        bad = diff & ~exempt
        assert not bad.any(), "level %d: %d non-exempt mismatches (first %s)" % (lvl, bad.sum(), np.argwhere(bad)[:3])
        exempt_diffs += int((diff & exempt).sum())
    # seven levels of fp32 radii: a few 1e-7 relative
    assert np.all(np.abs(radius_gpu.astype(np.float64) - xn) <= 4e-6 * xn + 1e-30)
    return exempt_diffs


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_polar_quantize_shuffled_slots(dtype):
    book, ref = polar_books(seed=3)
    n_tok, n_kv, bs = 1000, 3, 64
    rng = np.random.default_rng(7)
    num_blocks = (n_tok + bs - 1) // bs + 2
    slots = rng.permutation(num_blocks * bs)[:n_tok]
    slots[::97] = -1                              # skipped tokens
    cache = C.allocate_cache(book, num_blocks, n_kv)
    g = generator(11)
    scales = W.channel_scales(3, n_kv, (0.1, 10.0), 3, 30.0)
    k = W.gaussian_tokens(n_tok, scales, dtype, "cuda", g)
    v = W.gaussian_tokens(n_tok, scales, dtype, "cuda", g)
    k[5] = 0.0                                    # the zero vector: every angle atan2(0, 0) = 0
    quantize_into(book, cache, k, v, slots)
    hc = host_cache(cache)
    live = np.flatnonzero(slots >= 0)
    report = {}
    for which, x_t in (("k", k), ("v", v)):
        x = x_t[torch.as_tensor(live, device="cuda")].double().cpu().numpy().reshape(-1, 128)
        rec = rows_at(hc, which + "_codes", slots[live], n_kv, bs).reshape(len(x), -1)
        rad = rows_at(hc, which + "_norm", slots[live], n_kv, bs).reshape(-1)
        report[which + "_exempt_code_diffs"] = check_records(x, rec, rad, ref)
    codes = len(live) * n_kv * 127
    print("polar", dtype, report)
    assert all(n <= 1e-4 * codes + 4 for n in report.values())
    assert B.tq_get_last_device_error(book) == 0


@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_polar_decode_gqa_ragged_contexts_shuffled_blocks(group):
    n_kv = 2
    cfg = dict(n_kv=n_kv, block_size=64, dtype="bf16", seed=group, log_uniform=(0.1, 10.0), outliers=3,
               outlier_scale=30.0)
    book, ref = polar_books(seed=5)
    assert B.tq_decode_kernel_kind(book, n_kv * group, n_kv) == 0
    ctx = np.array([0, 1, 31, 33, 512, 513, 1500], dtype=np.int32)
    table, _ = W.block_layout(ctx, 64, True, seed=group)
    g = generator(40 + group)
    cache = fill_cache(book, cfg, ctx, table, g, chunk_tokens=700)
    q = W.queries(len(ctx), n_kv * group, torch.bfloat16, "cuda", g)
    out = decode(book, cache, q, table, ctx, 1500)
    pairs = [(b, h) for b in range(len(ctx)) for h in range(n_kv * group)]
    worst = check_decode(out, host_cache(cache), q, table, ctx, ref, pairs)
    print("polar decode G=%d: worst normalised error %.3g" % (group, worst))
    assert B.tq_get_last_device_error(book) == 0


def test_polar_decode_step_appends_then_attends():
    # tq_decode_step on a PolarQuant cache: the new token of every sequence is
    # coded at position ctx - 1, then the whole context (including it) is decoded
    n_kv, group, bs = 2, 4, 64
    cfg = dict(n_kv=n_kv, block_size=bs, dtype="bf16", seed=9, log_uniform=(0.1, 10.0), outliers=3,
               outlier_scale=30.0)
    book, ref = polar_books(seed=8)
    ctx = np.array([1, 200, 1025], dtype=np.int32)
    table, _ = W.block_layout(ctx, bs, True, seed=2)
    g = generator(77)
    prefill = np.maximum(ctx - 1, 0)
    cache = fill_cache(book, cfg, prefill, table, g, chunk_tokens=600)
    batch = len(ctx)
    k_new = W.gaussian_tokens(batch, W.channel_scales(9, n_kv, (0.1, 10.0), 3, 30.0), torch.bfloat16, "cuda", g)
    v_new = W.gaussian_tokens(batch, W.channel_scales(10, n_kv, (0.1, 10.0), 3, 30.0), torch.bfloat16, "cuda", g)
    q = W.queries(batch, n_kv * group, torch.bfloat16, "cuda", g)
    ws, nbytes = C.allocate_workspace(book, batch, n_kv * group, int(ctx.max()))
    out = torch.full((batch, n_kv * group, 128), float("nan"), device="cuda")
    table_t = torch.as_tensor(table, device="cuda")
    ctx_t = torch.as_tensor(ctx, device="cuda")
    B.tq_decode_step(book, k_new, v_new, B.TQ_BF16, q, B.TQ_BF16, batch, n_q_heads=n_kv * group, n_kv_heads=n_kv,
                     view=C.cache_view(book, cache), block_table=table_t, max_blocks=table.shape[1],
                     context_lens=ctx_t, max_context=int(ctx.max()), scale=0.0, out=out, workspace=ws,
                     workspace_bytes=nbytes)
    hc = host_cache(cache)
    slots = np.array([table[b, (c - 1) // bs] * bs + (c - 1) % bs for b, c in enumerate(ctx)])
    for which, x_t in (("k", k_new), ("v", v_new)):
        x = x_t.double().cpu().numpy().reshape(-1, 128)
        rec = rows_at(hc, which + "_codes", slots, n_kv, bs).reshape(len(x), -1)
        rad = rows_at(hc, which + "_norm", slots, n_kv, bs).reshape(-1)
        check_records(x, rec, rad, ref)
    pairs = [(b, h) for b in range(batch) for h in range(n_kv * group)]
    worst = check_decode(out.cpu().numpy(), hc, q, table, ctx, ref, pairs)
    print("polar decode step: worst normalised error %.3g" % worst)
    assert B.tq_get_last_device_error(book) == 0


def test_polar_cache_through_the_static_and_host_buffer_entry_points():
    # the allocation-free decode and the host-buffer step take a PolarQuant
    # handle like any other: their outputs equal the workspace decode's
    n_kv, group, bs = 2, 4, 64
    cfg = dict(n_kv=n_kv, block_size=bs, dtype="bf16", seed=12, log_uniform=(0.1, 10.0), outliers=3,
               outlier_scale=30.0)
    book, ref = polar_books(seed=12)
    ctx = np.array([300, 1100], dtype=np.int32)
    table, _ = W.block_layout(ctx, bs, True, seed=5)
    g = generator(90)
    cache = fill_cache(book, cfg, ctx, table, g, chunk_tokens=500)
    q = W.queries(2, n_kv * group, torch.bfloat16, "cuda", g)
    expect = decode(book, cache, q, table, ctx, int(ctx.max()))
    out = torch.full((2, n_kv * group, 128), float("nan"), device="cuda")
    table_t = torch.as_tensor(table, device="cuda")
    ctx_t = torch.as_tensor(ctx, device="cuda")
    B.tq_decode_attention_static(book, q, B.TQ_BF16, 2, n_kv * group, n_kv, C.cache_view(book, cache), table_t,
                                 table.shape[1], ctx_t, int(ctx.max()), 0.0, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), expect)
    # one host-buffer step appends a token per sequence and decodes; the same
    # step through device buffers on a copy of the cache gives the same output
    k_new = W.gaussian_tokens(2, W.channel_scales(3, n_kv, (0.1, 10.0), 3, 30.0), torch.bfloat16, "cuda", g)
    v_new = W.gaussian_tokens(2, W.channel_scales(4, n_kv, (0.1, 10.0), 3, 30.0), torch.bfloat16, "cuda", g)
    ctx2 = ctx + 1
    copy = {name: t.clone() for name, t in cache.items()}
    ws, nbytes = C.allocate_workspace(book, 2, n_kv * group, int(ctx2.max()))
    dev_out = torch.empty((2, n_kv * group, 128), device="cuda")
    ctx2_t = torch.as_tensor(ctx2, device="cuda")
    B.tq_decode_step(book, k_new, v_new, B.TQ_BF16, q, B.TQ_BF16, 2, n_kv * group, n_kv, C.cache_view(book, copy),
                     table_t, table.shape[1], ctx2_t, int(ctx2.max()), 0.0, dev_out, ws, nbytes)
    host_out = torch.empty((2, n_kv * group, 128)).pin_memory()
    hws = B.tq_decode_step_host_workspace_bytes(book, 2, n_kv * group, n_kv, int(ctx2.max()), B.TQ_BF16, B.TQ_BF16)
    hws_t = torch.empty(hws, dtype=torch.uint8, device="cuda")
    B.tq_decode_step_host(book, k_new.cpu().pin_memory(), v_new.cpu().pin_memory(), B.TQ_BF16,
                          q.cpu().pin_memory(), B.TQ_BF16, 2, n_kv * group, n_kv, C.cache_view(book, cache), table_t,
                          table.shape[1], torch.as_tensor(ctx2).pin_memory(), int(ctx2.max()), 0.0, host_out, hws_t,
                          hws, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert np.array_equal(host_out.numpy(), dev_out.cpu().numpy())
    assert B.tq_get_last_device_error(book) == 0
