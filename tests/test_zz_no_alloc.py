"""tq_decode_attention_static: decode attention for callers that cannot
allocate device memory (a runtime whose pool owns the whole GPU, or a loop
where an allocation and the synchronisation it may cause are not allowed).

It must give the results of tq_decode_attention with a caller workspace, on
two calls in a row (the built-in scratch keeps the previous call's contents),
and reject shapes whose scratch would not fit.  This file is collected last
so that a run stopping at the first failure has run every other test."""
import numpy as np
import pytest
import torch

from online_kv_cache_tq_gb300 import binding as B
from online_kv_cache_tq_gb300 import cache as C
from online_kv_cache_tq_gb300 import workloads as W

from parity_helpers import ATTN_TOL, books, check_decode, decode, fill_cache, generator, host_cache

pytestmark = pytest.mark.gpu


def _static_decode(book, cache, q, table, ctx, max_context):
    out = torch.full((q.shape[0], q.shape[1], 128), float("nan"), device="cuda")
    B.tq_decode_attention_static(book, q, B.TQ_BF16, q.shape[0], q.shape[1], cache["k_norm"].shape[1],
                                 C.cache_view(book, cache), torch.as_tensor(table, device="cuda"), table.shape[1],
                                 torch.as_tensor(ctx, device="cuda"), max_context, 0.0, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_static_scratch_matches_workspace_path_on_two_calls_in_a_row():
    cfg = dict(n_kv=4, block_size=64, dtype="bf16", seed=6, log_uniform=(0.1, 10.0), outliers=3,
               outlier_scale=30.0)
    book, ref = books(3, 3, 128, seed=2)
    g = generator(31)
    ctx = np.array([3000, 700, 1, 2049], dtype=np.int32)
    table, _ = W.block_layout(ctx, 64, True, seed=4)
    cache = fill_cache(book, cfg, ctx, table, g)
    hc = host_cache(cache)
    for call in range(2):                            # the second call reuses the scratch the first left
        q = W.queries(len(ctx), 16, torch.bfloat16, "cuda", g)
        expect = decode(book, cache, q, table, ctx, 3000)
        got = _static_decode(book, cache, q, table, ctx, 3000)
        assert np.all(np.isfinite(got))
        # same tolerance as the parity tests, normalised by the largest value norm in the cache
        assert np.max(np.abs(got - expect)) <= ATTN_TOL * float(hc["v_norm"].max())
        check_decode(got, hc, q, table, ctx, ref, [(b, h) for b in range(len(ctx)) for h in (0, 7, 15)])
    assert B.tq_get_last_device_error(book) == 0


def test_static_scratch_rejects_shapes_that_do_not_fit():
    book, _ = books()
    cache = C.allocate_cache(book, 2, 8)
    batch, n_q, max_context = 64, 64, 32768          # needs far more than the built-in scratch
    assert B.tq_decode_workspace_bytes(book, batch, n_q, max_context) > 16 << 20
    q = torch.zeros((batch, n_q, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((batch, n_q, 128), device="cuda")
    ctx = torch.zeros(batch, dtype=torch.int32, device="cuda")
    with pytest.raises(B.TQError) as err:
        B.tq_decode_attention_static(book, q, B.TQ_BF16, batch, n_q, 8, C.cache_view(book, cache), None, 1, ctx,
                                     max_context, 0.0, out)
    assert err.value.status == 5
