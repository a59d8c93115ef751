"""Whole-path oracle: codebook build, quantize-append into a paged cache, and
decode attention (test infrastructure only).

Bit split, 甲子光年 article §2 第二階段: a key budget of b bits per
coordinate is b-1 MSE bits plus the 1-bit QJL sketch; values use all their
bits for the MSE code and carry no sketch.  One R and one S serve keys,
values and every head (a reading; the pages draw one rotation per quantizer).
"""
import functools

import numpy as np

from . import attention, codebook, packing, polar, quantize, rotation


@functools.lru_cache(maxsize=None)
def _levels(d, bits):
    return codebook.lloyd_max(d, bits)


@functools.lru_cache(maxsize=None)
def _matrices(d, m, seed):
    return rotation.rotation_and_projection(d, m, seed)


def build(d=128, k_bits=3, v_bits=3, qjl_m=128, seed=0, norm_bits=32, codec="turboquant"):
    """The oracle's own R, S and codebooks for one configuration; norm_bits 16
    stores the norms (and the residual norm) as float16, 32 as float32.
    codec "polar": keys and values coded by PolarQuant (``polar``), no
    codebooks and no QJL; R is the same seeded draw."""
    if codec == "polar":
        rot, proj = _matrices(d, 0, seed)
        return {"codec": "polar", "d": d, "qjl_m": 0, "rot": rot, "proj": proj, "norm_dtype": np.float32}
    k_mse_bits = k_bits - 1 if qjl_m else k_bits
    rot, proj = _matrices(d, qjl_m, seed)
    k_levels, k_bounds = _levels(d, k_mse_bits)
    v_levels, v_bounds = _levels(d, v_bits)
    return {
        "d": d, "qjl_m": qjl_m, "rot": rot, "proj": proj,
        "k_bits": k_mse_bits, "v_bits": v_bits,
        "k_levels": k_levels, "k_bounds": k_bounds,
        "v_levels": v_levels, "v_bounds": v_bounds,
        "norm_dtype": np.float16 if norm_bits == 16 else np.float32,
    }


def _encode_polar(x, book, prefix):
    codes, radius, margins, y = polar.encode_vectors(x, book["rot"])
    return {prefix + "_codes": polar.pack(codes), prefix + "_norm": radius, "codes": codes, "margins": margins,
            "y": y}


def encode_keys(x, book):
    """Key rows: dict of packed codes, sign bits, norm, residual norm, plus the
    fp64 intermediates (unit rotated y, projected residual z) for acceptance."""
    if book.get("codec") == "polar":
        return _encode_polar(x, book, "k")
    nd = book.get("norm_dtype", np.float32)
    norm, y, codes = quantize.encode_mse(x, book["rot"], book["k_bounds"], nd)
    out = {"k_codes": packing.pack_planes(codes, book["k_bits"]), "k_norm": norm,
           "codes": codes, "y": y}
    if book["qjl_m"]:
        gamma, signs, z = quantize.encode_qjl(x, norm, codes, book["rot"], book["k_levels"], book["proj"], nd)
        out.update({"k_qjl": packing.pack_signs(signs), "k_rnorm": gamma, "signs": signs, "z": z})
    return out


def encode_values(x, book):
    """Value rows: packed codes and norm (plus fp64 intermediates)."""
    if book.get("codec") == "polar":
        return _encode_polar(x, book, "v")
    norm, y, codes = quantize.encode_mse(x, book["rot"], book["v_bounds"], book.get("norm_dtype", np.float32))
    return {"v_codes": packing.pack_planes(codes, book["v_bits"]), "v_norm": norm,
            "codes": codes, "y": y}


def field_bytes(book):
    """Bytes per (token, head) of each cache field."""
    d = book["d"]
    if book.get("codec") == "polar":
        return {"k_codes": polar.RECORD_BYTES, "k_norm": 4, "v_codes": polar.RECORD_BYTES, "v_norm": 4}
    nb = np.dtype(book.get("norm_dtype", np.float32)).itemsize
    out = {"k_codes": book["k_bits"] * d // 8, "k_norm": nb,
           "v_codes": book["v_bits"] * d // 8, "v_norm": nb}
    if book["qjl_m"]:
        out["k_qjl"] = book["qjl_m"] // 8
        out["k_rnorm"] = nb
    return out


def empty_cache(book, num_blocks, n_kv_heads, block_size):
    cache = {}
    for name, nbytes in field_bytes(book).items():
        if name == "v_codes" and book.get("codec") != "polar":
            cache[name] = np.zeros((num_blocks, n_kv_heads, book["v_bits"], book["d"], block_size // 8),
                                   dtype=np.uint8)
        elif name.endswith("norm"):
            cache[name] = np.zeros((num_blocks, n_kv_heads, block_size), dtype=book.get("norm_dtype", np.float32))
        else:
            cache[name] = np.zeros((num_blocks, n_kv_heads, block_size, nbytes), dtype=np.uint8)
    return cache


def append(cache, book, k, v, slots):
    """Quantize k, v [n_tokens][n_kv][d] and write them at ``slots`` (one slot
    per token; negative slots are skipped)."""
    num_blocks, n_kv, block_size = cache["k_norm"].shape
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_tok = k.shape[0]
    keys = encode_keys(k.reshape(n_tok * n_kv, -1), book)
    vals = encode_values(v.reshape(n_tok * n_kv, -1), book)
    polar_codec = book.get("codec") == "polar"
    live = [t for t in range(n_tok) if slots[t] >= 0]
    if not polar_codec:
        for h in range(n_kv):
            codes = vals["codes"].reshape(n_tok, n_kv, -1)[live, h]
            packing.write_value_codes(cache["v_codes"], codes, np.asarray(slots)[live], h)
    for name in field_bytes(book):
        if name == "v_codes" and not polar_codec:
            continue
        src = (keys if name.startswith("k_") else vals)[name]
        src = src.reshape(n_tok, n_kv, *src.shape[1:])
        flat = cache[name].reshape(num_blocks * n_kv * block_size, *cache[name].shape[3:])
        for t in range(n_tok):
            if slots[t] < 0:
                continue
            for h in range(n_kv):
                flat[packing.slot_index(slots[t], h, n_kv, block_size)] = src[t, h]
    return keys, vals


def decode(query, cache, block_table, context_lens, book, scale=None):
    """out [B][Hq][d] (fp64) and the per-(seq, head) normaliser max_t ||v_hat_t||."""
    query = np.asarray(query, dtype=np.float64)
    batch, n_q, d = query.shape
    n_kv = cache["k_norm"].shape[1]
    group = n_q // n_kv
    out = np.zeros((batch, n_q, d))
    vmax = np.zeros((batch, n_q))
    for b in range(batch):
        for h in range(n_q):
            out[b, h], vmax[b, h] = attention.decode_attention(
                query[b, h], cache, block_table[b], int(context_lens[b]), h // group, book, scale)
    return out, vmax
