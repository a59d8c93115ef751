"""Host logic of the benchmark's oracle leg (CPU only): the parity figures it
reports -- exempt and non-exempt code / sign disagreements, worst normalised
attention error -- must be zero for a cache the oracle wrote itself and must
count a mistake planted in that cache."""
import numpy as np

import bench
from oracle import attention, engine, packing, quantize


def _oracle_sample(bits=3, n_tok=40, n_kv=2, bs=64, seed=3):
    ref = engine.build(k_bits=bits, v_bits=bits, qjl_m=128, seed=0)
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((n_tok, n_kv, 128))
    v = rng.standard_normal((n_tok, n_kv, 128)) * 2.0
    cache = engine.empty_cache(ref, 1, n_kv, bs)
    slots = np.arange(n_tok)
    engine.append(cache, ref, k, v, slots)
    return ref, {"bits": bits, "qjl_m": 128, "seed": 0, "block_size": bs, "slots": slots, "k": k, "v": v,
                 "cache": cache}


def test_quant_parity_counts_nothing_on_the_oracles_own_cache():
    _, sample = _oracle_sample()
    rep = bench._quant_parity(sample)
    assert rep["vectors"] == 2 * 40 * 2
    assert rep["non_exempt_codes"] == 0 and rep["exempt_codes"] == 0
    assert rep["non_exempt_signs"] == 0 and rep["exempt_signs"] == 0


def test_quant_parity_counts_a_planted_code_and_sign():
    ref, sample = _oracle_sample()
    cache = sample["cache"]
    # a key coordinate far from every boundary: flip bit 0 of its code
    x = sample["k"][5, 1]
    _, y, _ = quantize.encode_mse(x[None, :], ref["rot"], ref["k_bounds"])
    j = int(np.argmax(quantize.boundary_distance(y, ref["k_bounds"])[0]))
    row = packing.slot_index(5, 1, 2, 64)
    flat = cache["k_codes"].reshape(-1, cache["k_codes"].shape[-1])
    flat[row, j // 8] ^= np.uint8(1 << (j % 8))
    rep = bench._quant_parity(sample)
    assert rep["non_exempt_codes"] == 1
    # the flipped code changes the residual the oracle recomputes, so some signs
    # may move too; a planted sign flip far from its hyperplane is counted on top
    _, sample2 = _oracle_sample()
    z = engine.encode_keys(sample2["k"][7, 0][None, :], ref)["z"][0]
    kk = int(np.argmax(np.abs(z)))
    flat2 = sample2["cache"]["k_qjl"].reshape(-1, 16)
    flat2[packing.slot_index(7, 0, 2, 64), kk // 8] ^= np.uint8(1 << (kk % 8))
    rep2 = bench._quant_parity(sample2)
    assert rep2["non_exempt_signs"] == 1 and rep2["non_exempt_codes"] == 0


def test_decode_parity_is_zero_for_oracle_outputs_and_sees_an_offset():
    ref, sample = _oracle_sample()
    cache = sample["cache"]
    rng = np.random.default_rng(9)
    q = rng.standard_normal((4, 128))
    out = np.stack([attention.decode_attention(q[h], cache, np.arange(1), 40, 1, ref)[0] for h in range(4)])
    cfg = {"k_bits": 3, "v_bits": 3, "qjl_m": 128, "seed": 0}
    item = {"b": 0, "kvh": 1, "ctx": 40, "cache": cache, "q": q, "out": out}
    assert bench._decode_parity_group((cfg, item)) < 1e-12
    vmax = attention.decode_attention(q[0], cache, np.arange(1), 40, 1, ref)[1]
    bad = dict(item, out=out + np.where(np.arange(128) == 3, 0.01 * vmax, 0.0))
    assert abs(bench._decode_parity_group((cfg, bad)) - 0.01) < 1e-9
