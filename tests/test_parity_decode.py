"""GPU decode attention vs the fp64 oracle, through the C ABI.

The oracle decodes the GPU's own packed cache (identical codes), so these
tests isolate the read path: scores, QJL correction, softmax, split-K merge
and back-rotation."""
import os

import numpy as np
import pytest
import torch

from online_kv_cache_tq_gb300 import binding as B
from online_kv_cache_tq_gb300 import cache as C
from online_kv_cache_tq_gb300 import workloads as W

from parity_helpers import (attn_pairs, books, check_decode, check_decode_groups, decode, fill_cache, generator,
                            host_cache, identity_table, run_boundary_groups, quantize_into)

pytestmark = pytest.mark.gpu


def test_single_head_fp32_every_output():
    cfg = W.CONFIGS["c1_single_head_parity"]
    book, ref = books(cfg["k_bits"], cfg["v_bits"], cfg["qjl_m"], cfg["seed"])
    g = generator(0)
    ctx = np.array([4096], dtype=np.int32)
    table = identity_table(1, 64)
    cache = fill_cache(book, cfg, ctx, table, g)
    q = W.queries(1, 1, torch.float32, "cuda", g)
    out = decode(book, cache, q, None, ctx, 4096)
    worst = check_decode(out, host_cache(cache), q, table, ctx, ref, [(0, 0)])
    print("c1 worst normalised error %.3g" % worst)
    assert B.tq_get_last_device_error(book) == 0


@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_gqa_ragged_contexts_shuffled_blocks(group):
    # contexts spanning 0, 1, partial and several 512-token chunks; shuffled pages
    n_kv = 2
    cfg = dict(n_kv=n_kv, block_size=64, dtype="bf16", seed=group, log_uniform=(0.1, 10.0), outliers=3,
               outlier_scale=30.0)
    book, ref = books(3, 3, 128, seed=1)
    assert B.tq_decode_kernel_kind(book, n_kv * group, n_kv) == 1      # tensor-core partials
    ctx = np.array([0, 1, 77, 512, 513, 1500, 2100], dtype=np.int32)
    table, _ = W.block_layout(ctx, 64, True, seed=group)
    g = generator(group)
    cache = fill_cache(book, cfg, ctx, table, g, chunk_tokens=1000)
    q = W.queries(len(ctx), n_kv * group, torch.bfloat16, "cuda", g)
    out = decode(book, cache, q, table, ctx, 2100)
    pairs = [(b, h) for b in range(len(ctx)) for h in range(n_kv * group)]
    check_decode(out, host_cache(cache), q, table, ctx, ref, pairs)
    assert B.tq_get_last_device_error(book) == 0


@pytest.mark.parametrize("group", [4, 8])
def test_long_contexts_over_few_groups_merge_per_query_head(group):
    # two sequences x two KV heads with contexts of 30 and 9 chunks: more
    # segments per group than the in-kernel merge takes and fewer groups than
    # SMs, so a merge launch with one CTA per query head follows the partials
    n_kv = 2
    cfg = dict(n_kv=n_kv, block_size=64, dtype="bf16", seed=20 + group, log_uniform=(0.1, 10.0), outliers=3,
               outlier_scale=30.0)
    book, ref = books(3, 3, 128, seed=6)
    ctx = np.array([15000, 4500], dtype=np.int32)
    table, _ = W.block_layout(ctx, 64, True, seed=group)
    plan = B.tq_decode_plan(book, 2, n_kv * group, n_kv, int(ctx.max()))
    assert plan["merge_in_partials"] == 0 and plan["merge_ctas"] == 2 * n_kv * group, plan
    g = generator(30 + group)
    cache = fill_cache(book, cfg, ctx, table, g, chunk_tokens=4000)
    q = W.queries(2, n_kv * group, torch.bfloat16, "cuda", g)
    out = decode(book, cache, q, table, ctx, int(ctx.max()))
    pairs = [(b, h) for b in range(2) for h in range(n_kv * group)]
    worst = check_decode(out, host_cache(cache), q, table, ctx, ref, pairs)
    print("per-head merge, G=%d: worst normalised error %.3g" % (group, worst))
    assert B.tq_get_last_device_error(book) == 0


@pytest.mark.parametrize("k_bits,v_bits,qjl", [(2, 1, 128), (5, 4, 128), (4, 2, 128), (2, 3, 0), (3, 2, 0)])
def test_bit_width_variants(k_bits, v_bits, qjl):
    # (4, 2, 128) and (3, 2, 0) have four MSE sign planes: key tiles built in two units, with and without the
    # QJL plane in the second
    cfg = dict(n_kv=1, block_size=64, dtype="bf16", seed=5, log_uniform=None, outliers=2, outlier_scale=20.0)
    book, ref = books(k_bits, v_bits, qjl, seed=2)
    ctx = np.array([1100, 300], dtype=np.int32)
    table, _ = W.block_layout(ctx, 64, False, seed=0)
    g = generator(k_bits)
    cache = fill_cache(book, cfg, ctx, table, g)
    q = W.queries(2, 4, torch.float32, "cuda", g)
    out = decode(book, cache, q, table, ctx, 1100)
    check_decode(out, host_cache(cache), q, table, ctx, ref, [(b, h) for b in range(2) for h in range(4)])


@pytest.mark.parametrize("block_size", [96, 1024])
def test_blocks_not_dividing_the_chunk_take_the_simt_kernel(block_size):
    # 512-token chunks cut through these blocks, which the tensor-core kernel
    # does not take: the SIMT partials kernel serves them
    cfg = dict(n_kv=2, block_size=block_size, dtype="bf16", seed=11, log_uniform=(0.1, 10.0), outliers=3,
               outlier_scale=30.0)
    book, ref = books(3, 3, 128, seed=4, block_size=block_size)
    assert B.tq_decode_kernel_kind(book, 8, 2) == 0
    ctx = np.array([1, 700, 1500], dtype=np.int32)
    table, _ = W.block_layout(ctx, block_size, True, seed=3)
    g = generator(block_size)
    cache = fill_cache(book, cfg, ctx, table, g, chunk_tokens=1000)
    q = W.queries(len(ctx), 8, torch.bfloat16, "cuda", g)
    out = decode(book, cache, q, table, ctx, 1500)
    check_decode(out, host_cache(cache), q, table, ctx, ref, [(b, h) for b in range(len(ctx)) for h in range(8)])
    assert B.tq_get_last_device_error(book) == 0


def test_staged_calls_match_the_one_call():
    cfg = dict(n_kv=2, block_size=64, dtype="bf16", seed=8, log_uniform=(0.1, 10.0), outliers=0,
               outlier_scale=1.0)
    book, _ = books(3, 3, 128, seed=5)
    ctx = np.array([700, 1300], dtype=np.int32)
    table, _ = W.block_layout(ctx, 64, True, seed=3)
    g = generator(11)
    cache = fill_cache(book, cfg, ctx, table, g)
    q = W.queries(2, 8, torch.bfloat16, "cuda", g)
    whole = decode(book, cache, q, table, ctx, 1300)
    ws, nbytes = C.allocate_workspace(book, 2, 8, 1300)
    out = torch.zeros((2, 8, 128), device="cuda")
    table_t = torch.as_tensor(table, device="cuda")
    ctx_t = torch.as_tensor(ctx, device="cuda")
    view = C.cache_view(book, cache)
    B.tq_decode_prepare(book, q, B.TQ_BF16, 2, 8, 1300, ws, nbytes)
    B.tq_decode_partials(book, 2, 8, 2, view, table_t, table.shape[1], ctx_t, 1300, 0.0, ws, nbytes)
    B.tq_decode_finish(book, 2, 8, ctx_t, 1300, table.shape[1], out, ws, nbytes)
    torch.cuda.synchronize()
    # the merge kernel and the in-place merge of the partials kernel order the
    # same additions differently: equal up to float rounding
    assert np.allclose(out.cpu().numpy(), whole, rtol=1e-5, atol=1e-6 * float(np.abs(whole).max()))
    # partials with an output: the in-place merge, bit for bit the one call
    out2 = torch.full_like(out, float("nan"))
    B.tq_decode_prepare(book, q, B.TQ_BF16, 2, 8, 1300, ws, nbytes)
    B.tq_decode_partials(book, 2, 8, 2, view, table_t, table.shape[1], ctx_t, 1300, 0.0, ws, nbytes, out=out2)
    torch.cuda.synchronize()
    assert np.array_equal(out2.cpu().numpy(), whole)


def test_custom_scale_and_device_errors():
    cfg = dict(n_kv=1, block_size=64, dtype="fp32", seed=3, log_uniform=None, outliers=0, outlier_scale=1.0)
    book, ref = books(3, 3, 128, seed=4)
    ctx = np.array([200], dtype=np.int32)
    table, _ = W.block_layout(ctx, 64, False, seed=0)
    g = generator(9)
    cache = fill_cache(book, cfg, ctx, table, g)
    q = W.queries(1, 1, torch.float32, "cuda", g)
    out = decode(book, cache, q, table, ctx, 200, scale=0.05)
    check_decode(out, host_cache(cache), q, table, ctx, ref, [(0, 0)], scale=0.05)
    # a block id outside the cache is skipped and recorded (code 2)
    bad = table.copy()
    bad[0, 1] = 1000
    decode(book, cache, q, bad, ctx, 200)
    assert B.tq_get_last_device_error(book) == 2
    # a context longer than max_context is clamped and recorded (code 3)
    decode(book, cache, q, table, np.array([300], dtype=np.int32), 200)
    assert B.tq_get_last_device_error(book) == 3
    assert B.tq_get_last_device_error(book) == 0


@pytest.mark.parametrize("group", [1, 4, 8])
def test_skipped_blocks_and_a_chunk_without_a_valid_slot(group):
    # Table entries outside the cache are skipped (and recorded): the output is
    # the attention over the remaining tokens, which the oracle gets from a table
    # with those entries taken out.  Sequence 1 loses every block of its second
    # 512-token chunk, so that chunk's item has no valid slot in any head.
    n_kv = 2
    cfg = dict(n_kv=n_kv, block_size=64, dtype="bf16", seed=20 + group, log_uniform=(0.1, 10.0), outliers=2,
               outlier_scale=20.0)
    book, ref = books(3, 3, 128, seed=7)
    assert B.tq_decode_kernel_kind(book, n_kv * group, n_kv) == 1      # tensor-core partials
    ctx = np.array([1300, 1100], dtype=np.int32)
    table, num_blocks = W.block_layout(ctx, 64, True, seed=group)
    g = generator(30 + group)
    cache = fill_cache(book, cfg, ctx, table, g, chunk_tokens=1000)
    q = W.queries(len(ctx), n_kv * group, torch.bfloat16, "cuda", g)
    bad = table.copy()
    bad[0, 3] = num_blocks + 5                   # one block past the cache
    bad[1, 8:16] = -1                            # tokens 512 .. 1023: the whole second chunk
    out = decode(book, cache, q, bad, ctx, 1300)
    assert B.tq_get_last_device_error(book) == 2
    assert np.all(np.isfinite(out))
    kept = np.full_like(table, -1)
    rows = [np.concatenate([table[0, :3], table[0, 4:21]]), np.concatenate([table[1, :8], table[1, 16:18]])]
    for b, r in enumerate(rows):
        kept[b, :len(r)] = r
    kept_ctx = np.array([1300 - 64, 1100 - 512], dtype=np.int32)
    pairs = [(b, h) for b in range(len(ctx)) for h in range(n_kv * group)]
    check_decode(out, host_cache(cache), q, kept, kept_ctx, ref, pairs)


def test_workspace_and_argument_checks():
    book, _ = books()
    cache = C.allocate_cache(book, 4, 1)
    view = C.cache_view(book, cache)
    q = torch.zeros((1, 1, 128), device="cuda")
    out = torch.zeros((1, 1, 128), device="cuda")
    ctx = torch.ones(1, dtype=torch.int32, device="cuda")
    need = B.tq_decode_workspace_bytes(book, 1, 1, 256)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.TQError) as err:
        B.tq_decode_attention(book, q, B.TQ_FP32, 1, 1, 1, view, None, 4, ctx, 256, 0.0, out, ws, need - 256)
    assert err.value.status == 5
    with pytest.raises(B.TQError) as err:
        B.tq_decode_attention(book, q, B.TQ_FP32, 1, 3, 1, view, None, 4, ctx, 256, 0.0, out, ws, need)
    assert err.value.status == 2                     # group of 3 is not built
    with pytest.raises(B.TQError) as err:
        B.tq_decode_attention(book, q, B.TQ_FP32, 1, 1, 2, view, None, 4, ctx, 256, 0.0, out, ws, need)
    assert err.value.status == 1                     # n_kv differs from the cache


def _full_size(name, seed, pick):
    cfg = W.CONFIGS[name]
    book, ref = books(cfg["k_bits"], cfg["v_bits"], cfg["qjl_m"], cfg["seed"])
    ctx = W.context_lengths(cfg, cfg["seed"])
    table, _ = W.block_layout(ctx, cfg["block_size"], cfg.get("shuffled_table", False), cfg["seed"])
    g = generator(seed)
    cache = fill_cache(book, cfg, ctx, table, g, chunk_tokens=8192)
    q = W.queries(cfg["batch"], cfg["n_q"], W.torch_dtype(cfg["dtype"]), "cuda", g)
    out = decode(book, cache, q, table, ctx, int(ctx.max()))
    assert np.all(np.isfinite(out))
    groups = pick(cfg, ctx)
    book_args = dict(k_bits=cfg["k_bits"], v_bits=cfg["v_bits"], qjl_m=cfg["qjl_m"], seed=cfg["seed"])
    worst = check_decode_groups(out, host_cache(cache), q, table, ctx, book_args, groups,
                                processes=min(16, os.cpu_count() or 1))
    print("%s worst normalised error %.3g over %d groups (%d query heads)" %
          (name, worst, len(groups), len(groups) * cfg["n_q"] // cfg["n_kv"]))
    assert B.tq_get_last_device_error(book) == 0
    return worst


def test_llama3_8b_decode_full_size():
    # 16 groups: every sequence once, KV heads spread, 64 query heads in all
    _full_size("c2_llama3_8b_decode", 21, lambda cfg, ctx: [(b, b % cfg["n_kv"]) for b in range(cfg["batch"])])


def test_long_context_full_size_every_head():
    # the one sequence's 8 KV heads: all 64 query heads
    _full_size("c4_long_context", 22, lambda cfg, ctx: [(0, h) for h in range(cfg["n_kv"])])


def test_llama3_70b_paged_full_size_run_boundaries():
    # every group that holds the first or the last chunk of a CTA's run in the
    # persistent tensor-core grid, where the item cursor enters and leaves
    # sequences and segments are merged across CTAs
    def pick(cfg, ctx):
        book = B.Codebook(k_bits=cfg["k_bits"], v_bits=cfg["v_bits"], qjl_m=cfg["qjl_m"], seed=cfg["seed"],
                          block_size=cfg["block_size"], device=0)
        plan = B.tq_decode_plan(book, cfg["batch"], cfg["n_q"], cfg["n_kv"], int(ctx.max()))
        assert plan["tensor_cores"] == 1 and plan["chunk_tokens"] == 512
        groups = run_boundary_groups(ctx, cfg["n_kv"], plan["partials_ctas"])
        assert len(groups) * cfg["n_q"] // cfg["n_kv"] >= 256
        return groups

    _full_size("c5_llama3_70b_paged", 23, pick)


@pytest.mark.parametrize("batch,n_kv,group", [(5, 2, 4), (130, 8, 1)])
def test_decode_step_equals_append_then_attention(batch, n_kv, group):
    # one call (fused append + query preparation and an early-started partials
    # kernel when batch * n_kv <= 1024, the tile quantizer otherwise), and the
    # same call with the step's inputs and output in pinned host memory, against
    # the two calls it stands for: identical caches and outputs, and the output
    # within tolerance of the oracle; sequence 0 has an empty context
    cfg = dict(n_kv=n_kv, block_size=64, dtype="bf16", seed=21, log_uniform=(0.1, 10.0), outliers=3,
               outlier_scale=30.0)
    book, ref = books(3, 3, 128, seed=6)
    rng = np.random.default_rng(batch)
    ctx = rng.integers(1, 1500, size=batch).astype(np.int32)
    ctx[0] = 0
    table, _ = W.block_layout(ctx, 64, True, seed=batch)
    g = generator(batch)
    cache = fill_cache(book, cfg, np.maximum(ctx - 1, 0), table, g, chunk_tokens=1000)
    n_q = n_kv * group
    k_new = W.gaussian_tokens(batch, W.channel_scales(3, n_kv, (0.1, 10.0), 3, 30.0), torch.bfloat16, "cuda", g)
    v_new = W.gaussian_tokens(batch, W.channel_scales(4, n_kv, (0.1, 10.0), 3, 30.0), torch.bfloat16, "cuda", g)
    q = W.queries(batch, n_q, torch.bfloat16, "cuda", g)
    slots = torch.as_tensor(np.array([W.slots_for(table[b], [int(ctx[b]) - 1], 64)[0] if ctx[b] > 0 else -1
                                      for b in range(batch)]), device="cuda")
    table_d = torch.as_tensor(table, device="cuda")
    ctx_d = torch.as_tensor(ctx, device="cuda")
    max_ctx = int(ctx.max())
    ws, nbytes = C.allocate_workspace(book, batch, n_q, max_ctx)
    outs, caches = [], []
    for mode in ("two_calls", "step", "host"):
        c = {name: t.clone() for name, t in cache.items()}
        view = C.cache_view(book, c)
        out = torch.full((batch, n_q, 128), float("nan"), device="cuda", dtype=torch.float32)
        if mode == "step":
            B.tq_decode_step(book, k_new, v_new, B.TQ_BF16, q, B.TQ_BF16, batch, n_q, n_kv, view, table_d,
                             table.shape[1], ctx_d, max_ctx, 0.0, out, ws, nbytes)
        elif mode == "host":
            hk, hv, hq = (t.cpu().pin_memory() for t in (k_new, v_new, q))
            hctx = torch.as_tensor(ctx).pin_memory()
            hout = torch.full((batch, n_q, 128), float("nan"), dtype=torch.float32).pin_memory()
            hbytes = B.tq_decode_step_host_workspace_bytes(book, batch, n_q, n_kv, max_ctx, B.TQ_BF16, B.TQ_BF16)
            assert hbytes > nbytes
            hws = torch.empty(hbytes, dtype=torch.uint8, device="cuda")
            with pytest.raises(B.TQError):       # a workspace without room for the staging area
                B.tq_decode_step_host(book, hk, hv, B.TQ_BF16, hq, B.TQ_BF16, batch, n_q, n_kv, view, table_d,
                                      table.shape[1], hctx, max_ctx, 0.0, hout, hws, 1024)
            B.tq_decode_step_host(book, hk, hv, B.TQ_BF16, hq, B.TQ_BF16, batch, n_q, n_kv, view, table_d,
                                  table.shape[1], hctx, max_ctx, 0.0, hout, hws, hbytes)
            torch.cuda.synchronize()
            out.copy_(hout)
        else:
            B.tq_quantize_append(book, k_new, v_new, B.TQ_BF16, batch, n_kv, slots, view)
            B.tq_decode_attention(book, q, B.TQ_BF16, batch, n_q, n_kv, view, table_d, table.shape[1], ctx_d,
                                  max_ctx, 0.0, out, ws, nbytes)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
        caches.append({name: t.cpu() for name, t in c.items()})
    for other in (1, 2):
        for name in caches[0]:
            assert torch.equal(caches[0][name], caches[other][name]), name
        assert np.array_equal(outs[0], outs[other])
    pairs = [(0, 0)] + attn_pairs(batch, n_q, 12, seed=batch)
    check_decode(outs[1], host_cache(caches[1]), q, table, ctx, ref, pairs)
    assert B.tq_get_last_device_error(book) == 0


def test_every_context_empty_gives_zero_rows():
    # no chunk at all (max_context 0): the in-place merging launch still writes the zero outputs
    book, _ = books(3, 3, 128, seed=1)
    cache = C.allocate_cache(book, 3, 2)           # one block per sequence (identity layout)
    q = W.queries(3, 8, torch.bfloat16, "cuda", generator(1))
    for max_context in (0, 700):
        out = decode(book, cache, q, None, np.zeros(3, dtype=np.int32), max_context)
        assert np.all(out == 0.0)
    assert B.tq_get_last_device_error(book) == 0


@pytest.mark.parametrize("k_bits,v_bits,norm_bits,block_size,group", [
    (4, 2, 16, 64, 8),      # the 4-bit-key build with float16 norms
    (4, 2, 32, 64, 8),      # ... with float32 norms
    (3, 3, 32, 32, 8),      # 3/3 bits in 32-token blocks: the build that reads the shape from the arguments
    (3, 3, 16, 128, 4),     # ... 128-token blocks, float16 norms
    (4, 2, 32, 256, 8),     # ... 256-token blocks
])
def test_fixed_and_run_time_shape_builds(k_bits, v_bits, norm_bits, block_size, group):
    # every tensor-core build the launcher picks (widths, norm width and block
    # size folded in, or read from the arguments) against the oracle, over
    # ragged contexts and shuffled blocks
    n_kv = 2
    cfg = dict(n_kv=n_kv, block_size=block_size, dtype="bf16", seed=60 + block_size, log_uniform=(0.1, 10.0),
               outliers=3, outlier_scale=30.0)
    book, ref = books(k_bits, v_bits, 128, seed=9, block_size=block_size, norm_bits=norm_bits)
    assert B.tq_decode_kernel_kind(book, n_kv * group, n_kv) == 1
    ctx = np.array([0, 1, 77, 513, 1500], dtype=np.int32)
    table, _ = W.block_layout(ctx, block_size, True, seed=block_size)
    g = generator(70 + block_size)
    cache = fill_cache(book, cfg, ctx, table, g, chunk_tokens=1000)
    q = W.queries(len(ctx), n_kv * group, torch.bfloat16, "cuda", g)
    out = decode(book, cache, q, table, ctx, 1500)
    worst = check_decode(out, host_cache(cache), q, table, ctx, ref,
                         [(b, h) for b in range(len(ctx)) for h in range(n_kv * group)])
    print("K%d V%d, %d-bit norms, %d-token blocks, G=%d: worst normalised error %.3g"
          % (k_bits, v_bits, norm_bits, block_size, group, worst))
    assert B.tq_get_last_device_error(book) == 0


@pytest.mark.parametrize("norm_bits", [32, 16])
def test_extreme_magnitudes_and_sharp_softmax(norm_bits):
    # tokens scaled log-uniformly over 1e-3 .. 1e3 (and a few zero vectors), queries 20x larger than the rest
    # of the tests (scores in the hundreds: a sharp softmax): the piece scales of the query and weight operands
    # and the running max of the merge against the oracle
    n_kv, group, bs = 2, 8, 64
    book, ref = books(3, 3, 128, seed=13, norm_bits=norm_bits)
    ctx = np.array([700, 1500], dtype=np.int32)
    table, _ = W.block_layout(ctx, bs, True, seed=13)
    num_blocks = int(table.max()) + 1
    cache = C.allocate_cache(book, num_blocks, n_kv)
    g = generator(131)
    rng = np.random.default_rng(131)
    ones = np.ones((n_kv, 128))
    for b, length in enumerate(ctx):
        n = int(length)
        factors = np.exp(rng.uniform(np.log(1e-3), np.log(1e3), size=(n, n_kv, 1)))
        factors[rng.choice(n, size=3, replace=False)] = 0.0          # zero vectors
        f = torch.as_tensor(factors, dtype=torch.float32, device="cuda")
        k = (W.gaussian_tokens(n, ones, torch.float32, "cuda", g) * f).to(torch.bfloat16)
        v = (W.gaussian_tokens(n, ones, torch.float32, "cuda", g) * f).to(torch.bfloat16)
        quantize_into(book, cache, k, v, W.slots_for(table[b], np.arange(n), bs))
    q = (W.queries(2, n_kv * group, torch.float32, "cuda", g) * 20.0).to(torch.bfloat16)
    out = decode(book, cache, q, table, ctx, int(ctx.max()))
    worst = check_decode(out, host_cache(cache), q, table, ctx, ref,
                         [(b, h) for b in range(2) for h in range(n_kv * group)])
    print("extreme magnitudes, %d-bit norms: worst normalised error %.3g" % (norm_bits, worst))
    assert B.tq_get_last_device_error(book) == 0


@pytest.mark.parametrize("group", [4, 8])
def test_sixteen_bit_norms_decode(group):
    # a cache with float16 norms (102 bytes per token-head at 3/3 bits), ragged
    # contexts over shuffled blocks; the oracle decodes the GPU's cache
    n_kv = 2
    cfg = dict(n_kv=n_kv, block_size=64, dtype="bf16", seed=group + 40, log_uniform=(0.1, 10.0), outliers=3,
               outlier_scale=30.0)
    book, ref = books(3, 3, 128, seed=3, norm_bits=16)
    assert B.tq_decode_kernel_kind(book, n_kv * group, n_kv) == 1
    ctx = np.array([1, 300, 512, 1700, 2600], dtype=np.int32)
    table, _ = W.block_layout(ctx, 64, True, seed=group)
    g = generator(group + 40)
    cache = fill_cache(book, cfg, ctx, table, g, chunk_tokens=1000)
    q = W.queries(len(ctx), n_kv * group, torch.bfloat16, "cuda", g)
    out = decode(book, cache, q, table, ctx, 2600)
    worst = check_decode(out, host_cache(cache), q, table, ctx, ref,
                         [(b, h) for b in range(len(ctx)) for h in range(n_kv * group)])
    print("fp16 norms, G=%d: worst normalised error %.3g" % (group, worst))
    assert B.tq_get_last_device_error(book) == 0


def test_decode_plan_for_the_workloads():
    # the launch plan: the 8B layer merges in the partials kernel (128 groups,
    # fewer than CTAs, about four segments each), the 70B paged batch (512
    # groups) takes a merge launch with a CTA per group, and the long-context
    # layer (8 groups of about 40 segments) a merge launch with a CTA per
    # query head; its 4-bit-key layout also fits two CTAs per SM with 512-token
    # items (the output-exchange buffer lies inside the score buffer)
    expect = {"c2_llama3_8b_decode": (1, 512, 0), "c5_llama3_70b_paged": (0, 512, 512),
              "c4_long_context": (0, 512, 64)}
    for name, (fused, chunk, merge_ctas) in expect.items():
        cfg = W.CONFIGS[name]
        book = B.Codebook(k_bits=cfg["k_bits"], v_bits=cfg["v_bits"], qjl_m=cfg["qjl_m"], seed=cfg["seed"],
                          block_size=cfg["block_size"], device=0)
        ctx = W.context_lengths(cfg, cfg["seed"])
        plan = B.tq_decode_plan(book, cfg["batch"], cfg["n_q"], cfg["n_kv"], int(ctx.max()))
        assert plan["tensor_cores"] == 1
        assert (plan["merge_in_partials"], plan["chunk_tokens"], plan["merge_ctas"]) == (fused, chunk, merge_ctas), \
            (name, plan)
        assert 0 < plan["partials_ctas"] <= 2 * torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("batch", [2, 400])
def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_correct(batch):
    # the test aid withholds one MMA commit in the first CTA of the tensor-core
    # kernel: that CTA's builders wait the one-second limit, the CTA drains its
    # copies and MMAs and stops, the call ends with device error 4; with the
    # aid off the same handle decodes correctly again.  batch 2 merges in the
    # partials kernel, batch 400 (more groups than CTAs) in a merge launch,
    # which must reject the stale segment records the stopped CTA left.
    cfg = dict(n_kv=1, block_size=64, dtype="bf16", seed=batch, log_uniform=(0.1, 10.0), outliers=3,
               outlier_scale=30.0)
    book, ref = books(3, 3, 128, seed=14)
    rng = np.random.default_rng(batch)
    ctx = rng.integers(600, 1400, size=batch).astype(np.int32)
    table, _ = W.block_layout(ctx, 64, True, seed=batch)
    g = generator(batch + 1)
    cache = fill_cache(book, cfg, ctx, table, g, chunk_tokens=2000)
    q = W.queries(batch, 4, torch.bfloat16, "cuda", g)
    plan = B.tq_decode_plan(book, batch, 4, 1, int(ctx.max()))
    assert plan["merge_in_partials"] == (1 if batch == 2 else 0)
    B.tq_debug_withhold_commit(book, True)
    decode(book, cache, q, table, ctx, int(ctx.max()))
    assert B.tq_get_last_device_error(book) == 4
    B.tq_debug_withhold_commit(book, False)
    out = decode(book, cache, q, table, ctx, int(ctx.max()))
    assert B.tq_get_last_device_error(book) == 0
    pairs = [(b, h) for b in range(batch) for h in range(4)] if batch <= 8 else attn_pairs(batch, 4, 24, seed=3)
    check_decode(out, host_cache(cache), q, table, ctx, ref, pairs)


def test_prefill_at_four_bits_decode_at_three_bits():
    # the prompt's tokens in a 4-bit cache (3 MSE bits + QJL for keys, 4-bit
    # values), the generated ones in a 3-bit cache, one softmax over both; the
    # handles share the seed (one R, one S).  Sequences with an empty part, and
    # one with both parts empty.
    n_kv, g4 = 2, 4
    cfg = dict(n_kv=n_kv, block_size=64, dtype="bf16", seed=31, log_uniform=(0.1, 10.0), outliers=3,
               outlier_scale=30.0)
    book_p, ref_p = books(4, 4, 128, seed=6)
    book_d, ref_d = books(3, 3, 128, seed=6, norm_bits=16)
    pre = np.array([700, 0, 1500, 300, 0], dtype=np.int32)
    gen = np.array([5, 40, 0, 130, 0], dtype=np.int32)
    table_p, _ = W.block_layout(pre, 64, True, seed=1)
    table_d, _ = W.block_layout(gen, 64, True, seed=2)
    g = generator(31)
    cache_p = fill_cache(book_p, cfg, pre, table_p, g, chunk_tokens=1000)
    cache_d = fill_cache(book_d, cfg, gen, table_d, g, chunk_tokens=1000)
    batch, n_q = len(pre), n_kv * g4
    q = W.queries(batch, n_q, torch.bfloat16, "cuda", g)
    tp, td = (torch.as_tensor(t, device="cuda") for t in (table_p, table_d))
    lp, ld = (torch.as_tensor(c, device="cuda") for c in (pre, gen))
    first = B.context_part(book_p, C.cache_view(book_p, cache_p), tp, table_p.shape[1], lp, int(pre.max()))
    second = B.context_part(book_d, C.cache_view(book_d, cache_d), td, table_d.shape[1], ld, int(gen.max()))
    nbytes = B.tq_decode_parts_workspace_bytes(first, second, batch, n_q)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.full((batch, n_q, 128), float("nan"), device="cuda")
    B.tq_decode_attention_parts(first, second, q, B.TQ_BF16, batch, n_q, n_kv, 0.0, out, ws, nbytes)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    hp, hd = host_cache(cache_p), host_cache(cache_d)
    qn = q.double().cpu().numpy()
    from oracle import attention
    worst = 0.0
    for b in range(batch):
        for h in range(n_q):
            if pre[b] + gen[b] == 0:
                assert np.all(got[b, h] == 0.0)
                continue
            expect, vmax = attention.decode_attention_parts(
                qn[b, h], [(hp, table_p[b], int(pre[b]), h // g4, ref_p), (hd, table_d[b], int(gen[b]), h // g4, ref_d)])
            err = np.max(np.abs(got[b, h] - expect)) / vmax
            assert err <= 1e-3, (b, h, err)
            worst = max(worst, err)
    print("two-part decode: worst normalised error %.3g" % worst)
    assert B.tq_get_last_device_error(book_p) == 0
    # handles with different seeds (different R) are rejected
    other, _ = books(3, 3, 128, seed=7)
    bad = B.context_part(other, C.cache_view(book_d, cache_d), td, table_d.shape[1], ld, int(gen.max()))
    with pytest.raises(B.TQError):
        B.tq_decode_attention_parts(first, bad, q, B.TQ_BF16, batch, n_q, n_kv, 0.0, out, ws, nbytes)
