"""GPU quantize-append vs the fp64 oracle, through the C ABI.

Up to 1024 vectors per tensor take the per-vector kernel; larger appends the
tcgen05 tile quantizer (bf16 inputs through TMA, fp32 inputs split into bf16
hi/lo operands by converter warps)."""
import numpy as np
import pytest
import torch

from online_kv_cache_tq_gb300 import binding as B
from online_kv_cache_tq_gb300 import cache as C
from online_kv_cache_tq_gb300 import workloads as W

from parity_helpers import books, check_append, generator, host_cache, quantize_into

pytestmark = pytest.mark.gpu


def test_single_head_fp32_outliers_every_vector():
    # 4096 fp32 keys/values, 4 channels x20 (seeded separately), b = 3
    cfg = W.CONFIGS["c1_single_head_parity"]
    book, ref = books(cfg["k_bits"], cfg["v_bits"], cfg["qjl_m"], cfg["seed"])
    g = generator(0)
    k = W.gaussian_tokens(4096, W.channel_scales(0, 1, None, 4, 20.0), torch.float32, "cuda", g)
    v = W.gaussian_tokens(4096, W.channel_scales(1, 1, None, 4, 20.0), torch.float32, "cuda", g)
    cache = C.allocate_cache(book, 4096 // 64, 1)
    slots = np.arange(4096)
    quantize_into(book, cache, k, v, slots)
    rep = check_append(book, ref, cache, k, v, slots)
    print("c1 fp32 append", rep)
    assert rep["vectors"] == 4096
    assert B.tq_get_last_device_error(book) == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("k_bits,v_bits", [(2, 2), (3, 3), (4, 4), (5, 1), (4, 2)])
def test_tile_quantizer_gqa_ragged_shuffled_slots(k_bits, v_bits, dtype):
    # shuffled slots: value codes take the bit-by-bit path; fp32 inputs are
    # split into bf16 hi/lo operands on the tensor cores (three products)
    book, ref = books(k_bits, v_bits, 128, seed=3)
    n_tok, n_kv = 1001, 3                 # 3003 vectors: 24 tiles of 128 and a ragged tail
    g = generator(k_bits * 10 + v_bits)
    scales = W.channel_scales(5, n_kv, (0.1, 10.0), 3, 30.0)
    k = W.gaussian_tokens(n_tok, scales, dtype, "cuda", g)
    v = W.gaussian_tokens(n_tok, scales[::-1].copy(), dtype, "cuda", g)
    num_blocks = 20
    slots = np.random.default_rng(1).permutation(num_blocks * 64)[:n_tok]
    cache = C.allocate_cache(book, num_blocks, n_kv)
    quantize_into(book, cache, k, v, slots)
    print(check_append(book, ref, cache, k, v, slots))
    assert B.tq_get_last_device_error(book) == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_qjl_off_and_separate_k_v_calls(dtype):
    book, ref = books(3, 2, 0, seed=9)
    g = generator(2)
    k = W.gaussian_tokens(300, np.ones((2, 128)), dtype, "cuda", g)
    v = W.gaussian_tokens(300, np.ones((2, 128)), dtype, "cuda", g)
    cache = C.allocate_cache(book, 5, 2)
    assert "k_qjl" not in cache
    slots = np.arange(300)
    quantize_into(book, cache, k, None, slots)
    quantize_into(book, cache, None, v, slots)
    check_append(book, ref, cache, k, v, slots)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_zero_vectors_negative_and_out_of_range_slots(dtype):
    book, ref = books(3, 3, 128, seed=0)
    g = generator(4)
    k = W.gaussian_tokens(40, np.ones((2, 128)), dtype, "cuda", g)
    v = W.gaussian_tokens(40, np.ones((2, 128)), dtype, "cuda", g)
    k[5] = 0.0
    v[6] = 0.0
    cache = C.allocate_cache(book, 1, 2)
    for name in cache:
        cache[name].fill_(0xAB if cache[name].dtype == torch.uint8 else 7.0)
    slots = np.full(40, -1)
    slots[:10] = np.arange(10)
    slots[3] = -1                         # skipped silently
    slots[10] = 64 + 5                    # beyond the one-block cache: skipped and recorded
    quantize_into(book, cache, k, v, slots)
    assert B.tq_get_last_device_error(book) == 1
    assert B.tq_get_last_device_error(book) == 0       # cleared by the read
    valid = np.array([t for t in range(40) if 0 <= slots[t] < 64])
    check_append(book, ref, cache, k, v, slots, sample=valid)
    hc = {n: t.cpu() for n, t in cache.items()}
    assert torch.all(hc["k_codes"][0, :, 3] == 0xAB) and torch.all(hc["v_norm"][0, :, 3] == 7.0)
    # untouched value-code bits (token offset 3, and offsets 10..63) keep their old contents
    vbits = np.unpackbits(hc["v_codes"].numpy()[0], axis=-1, bitorder="little")   # [head][plane][dim][64]
    assert np.all(vbits[..., 3] == 1) and np.all(vbits[..., 10:] == np.unpackbits(np.uint8(0xAB), bitorder="little")[
        np.arange(10, 64) % 8])


@pytest.mark.parametrize("n_tok", [64, 1000, 2048])
def test_bf16_contiguous_prefill_and_partial_blocks(n_tok):
    # contiguous slots from offset 0 (whole 32-token words) and an offset start
    # (a partial first and last word): both value-code paths, then a second
    # append that overwrites part of the first
    book, ref = books(3, 3, 128, seed=7)
    n_kv = 4
    g = generator(n_tok)
    scales = W.channel_scales(2, n_kv, (0.1, 10.0), 3, 30.0)
    num_blocks = (n_tok + 100) // 64 + 2
    cache = C.allocate_cache(book, num_blocks, n_kv)
    for start in (0, 37):
        k = W.gaussian_tokens(n_tok, scales, torch.bfloat16, "cuda", g)
        v = W.gaussian_tokens(n_tok, scales, torch.bfloat16, "cuda", g)
        slots = np.arange(start, start + n_tok)
        quantize_into(book, cache, k, v, slots)
        check_append(book, ref, cache, k, v, slots)
    assert B.tq_get_last_device_error(book) == 0


def test_empty_append_is_a_no_op():
    book, _ = books()
    cache = C.allocate_cache(book, 1, 1)
    view = C.cache_view(book, cache)
    B.tq_quantize_append(book, None, None, B.TQ_BF16, 0, 1, None, view)
    with pytest.raises(B.TQError):
        B.tq_quantize_append(book, None, None, B.TQ_BF16, 1, 1, None, view)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_prefill_full_size_sampled(bits):
    # 32768 tokens x 8 KV heads, Student-t(3) channels, in the benchmark's launch shape
    cfg = W.CONFIGS["c3_prefill_quantize"]
    book, ref = books(bits, bits, 128, seed=0)
    g = generator(bits)
    k = W.student_t_tokens(cfg["tokens"], cfg["n_kv"], cfg["student_t_channels"], torch.bfloat16, "cuda", g, 0)
    v = W.student_t_tokens(cfg["tokens"], cfg["n_kv"], cfg["student_t_channels"], torch.bfloat16, "cuda", g, 1)
    cache = C.allocate_cache(book, cfg["tokens"] // 64, cfg["n_kv"])
    slots = np.arange(cfg["tokens"])
    quantize_into(book, cache, k, v, slots)
    sample = np.random.default_rng(bits).choice(cfg["tokens"], size=400, replace=False)
    sample = np.concatenate([sample, [0, cfg["tokens"] - 1]])
    rep = check_append(book, ref, cache, k, v, slots, sample=sample)
    print("prefill bits=%d" % bits, rep)
    assert B.tq_get_last_device_error(book) == 0


@pytest.mark.parametrize("dtype,n_tok", [(torch.bfloat16, 1001), (torch.float32, 300), (torch.bfloat16, 40)])
def test_sixteen_bit_norms(dtype, n_tok):
    # float16 norms on every append path (tile quantizers and the per-vector
    # one): norms within half an ulp, the residual taken against the stored
    # float16 norm (the oracle recomputes it from the GPU's codes and norm)
    book, ref = books(3, 3, 128, seed=8, norm_bits=16)
    n_kv = 3
    g = generator(n_tok)
    scales = W.channel_scales(6, n_kv, (0.1, 10.0), 3, 30.0)
    k = W.gaussian_tokens(n_tok, scales, dtype, "cuda", g)
    v = W.gaussian_tokens(n_tok, scales, dtype, "cuda", g)
    num_blocks = (n_tok + 63) // 64 + 1
    cache = C.allocate_cache(book, num_blocks, n_kv)
    assert cache["k_norm"].dtype == torch.float16
    slots = np.random.default_rng(n_tok).permutation(num_blocks * 64)[:n_tok]
    quantize_into(book, cache, k, v, slots)
    print(check_append(book, ref, cache, k, v, slots))
    assert B.tq_get_last_device_error(book) == 0


@pytest.mark.parametrize("norm_bits,dtype", [(32, torch.bfloat16), (16, torch.float32)])
def test_reconstruction_error_monitor(norm_bits, dtype):
    # the monitor's sums against the oracle's fp64 reconstruction n R^T c[code]
    # of the GPU's own codes and stored norms, for keys and values; a second
    # call adds to the first; a skipped slot is not counted
    from oracle import packing, quantize
    book, ref = books(3, 3, 128, seed=12, norm_bits=norm_bits)
    n_tok, n_kv = 700, 2
    g = generator(70 + norm_bits)
    scales = W.channel_scales(3, n_kv, (0.1, 10.0), 3, 30.0)
    k = W.gaussian_tokens(n_tok, scales, dtype, "cuda", g)
    v = W.gaussian_tokens(n_tok, scales, dtype, "cuda", g)
    cache = C.allocate_cache(book, 12, n_kv)
    slots = np.arange(n_tok)
    slots[5] = -1
    slot_t = quantize_into(book, cache, k, v, slots)
    view = C.cache_view(book, cache)
    hc = host_cache(cache)
    live = slots >= 0
    for which, x_t, name in ((0, k, "k"), (1, v, "v")):
        stats = torch.zeros(4, dtype=torch.float64, device="cuda")
        code = B.TQ_BF16 if dtype == torch.bfloat16 else B.TQ_FP32
        B.tq_reconstruction_error(book, x_t, code, which, n_tok, n_kv, slot_t, view, stats)
        B.tq_reconstruction_error(book, x_t, code, which, n_tok, n_kv, slot_t, view, stats)
        got = stats.cpu().numpy() / 2.0
        x = x_t.double().cpu().numpy()[live].reshape(-1, 128)
        rows = np.stack([packing.slot_index(slots[live], h, n_kv, 64) for h in range(n_kv)], axis=1).reshape(-1)
        if name == "k":
            codes = packing.unpack_planes(hc["k_codes"].reshape(-1, hc["k_codes"].shape[-1])[rows], ref["k_bits"], 128)
        else:
            codes = np.stack([packing.read_value_codes(hc["v_codes"], slots[live], h) for h in range(n_kv)],
                             axis=1).reshape(-1, 128)
        norm = hc[name + "_norm"].reshape(-1)[rows]
        err = np.linalg.norm(x - quantize.reconstruct_mse(norm, codes, ref["rot"], ref[name + "_levels"]), axis=1)
        expect = np.array([err.sum(), (err ** 2).sum(), (x * x).sum(), len(x)])
        assert got[3] == expect[3] == (n_tok - 1) * n_kv
        assert np.allclose(got[:3], expect[:3], rtol=1e-5), (name, got, expect)
        print(name, "mean error %.4g, relative squared error %.4g" % (got[0] / got[3], got[1] / got[2]))
    assert B.tq_get_last_device_error(book) == 0
