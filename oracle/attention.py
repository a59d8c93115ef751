"""Decode attention over the compressed cache (test infrastructure only).

* Inner-product estimate, 甲子光年 article §2 第二階段 (the stage-1 inner
  product is biased, the 1-bit QJL sketch of the residual makes the sum
  unbiased) and intelliparadigm.com §2.1.2 / §2.2 theorem 2 (the estimate's
  expectation equals the true inner product).  Reading: the asymmetric QJL
  estimator -- the query is projected but not quantized --

      <q, k> ~= <q, k_mse> + gamma * sqrt(pi/2) / m * <S q, 2 bits - 1>,

  exactly unbiased because E[<g, q> sign(<g, r>)] = sqrt(2/pi) <q, r> / ||r||
  for g ~ N(0, I).  The symmetric "C sign(Aq) sign(Ae)" form printed on the
  intelliparadigm page cannot be unbiased (its mean is not linear in <q, e>)
  and is not used.
* Attention: scaled dot-product softmax over every cached token of the
  sequence (a decode step sees its whole context), scale 1/sqrt(d) unless
  given; values are the stage-1 reconstructions n_v R^T c_v[code].  The query
  is not compressed (seo-farm page §4).  This oracle works in the original
  space; rotation invariance (seo-farm §2, R^T R = I) is what lets a kernel
  work in the rotated space instead.
* A PolarQuant cache (``polar``) holds reconstructible keys and values with no
  QJL term: the same softmax over <q, x_hat_k> applied to x_hat_v.
"""
import math

import numpy as np

from . import packing, polar
from .quantize import reconstruct_mse


def qjl_estimate(query, gamma32, signs, proj):
    """gamma * sqrt(pi/2) / m * <S q, 2 s - 1> for every cached token."""
    proj = np.asarray(proj, dtype=np.float64)
    m = proj.shape[0]
    sq = proj @ np.asarray(query, dtype=np.float64)
    pm = 2.0 * np.asarray(signs, dtype=np.float64) - 1.0
    return gamma32.astype(np.float64) * math.sqrt(math.pi / 2.0) / m * (pm @ sq)


def attend(query, khat, qjl_term, vhat, scale):
    """softmax(scale * (khat q + qjl_term)) @ vhat, all fp64."""
    logits = scale * (np.asarray(khat) @ np.asarray(query, dtype=np.float64) + qjl_term)
    logits = logits - np.max(logits)
    weights = np.exp(logits)
    weights /= np.sum(weights)
    return weights @ np.asarray(vhat)


def read_sequence(cache, table_row, length, head, block_size, polar_codec=False):
    """Rows of every token-major cache field, and the value codes, for tokens
    0..length-1 of one sequence/head (value codes as ``v_code_values``; a
    PolarQuant cache keeps its value records token-major)."""
    n_kv = cache["k_norm"].shape[1]
    pos = np.arange(length, dtype=np.int64)
    blocks = np.asarray(table_row, dtype=np.int64)[pos // block_size]
    rows = (blocks * n_kv + head) * block_size + pos % block_size
    out = {}
    for name, arr in cache.items():
        if name == "v_codes" and not polar_codec:
            out["v_code_values"] = packing.read_value_codes(arr, blocks * block_size + pos % block_size, head)
            continue
        flat = arr.reshape(arr.shape[0] * arr.shape[1] * arr.shape[2], -1)
        out[name] = flat[rows]
    return out


def _polar_rows(cache, table_row, length, kv_head, book):
    """Reconstructed keys and values [length][d] of a PolarQuant cache."""
    rows = read_sequence(cache, table_row, length, kv_head, cache["k_norm"].shape[2], polar_codec=True)
    khat = polar.reconstruct(polar.unpack(rows["k_codes"]), rows["k_norm"].reshape(-1), book["rot"])
    vhat = polar.reconstruct(polar.unpack(rows["v_codes"]), rows["v_norm"].reshape(-1), book["rot"])
    return khat, vhat


def decode_attention_heads(queries, cache, table_row, length, kv_head, book, scale=None):
    """Outputs [H][d] of several query heads that read the same sequence and
    KV head (a GQA group), and the normaliser max_t ||v_hat_t||: the same
    arithmetic as ``decode_attention`` per head, with the cached keys and
    values reconstructed once for the group."""
    d = book["rot"].shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if book.get("codec") == "polar":
        khat, vhat = _polar_rows(cache, table_row, length, kv_head, book)
        outs = [attend(q, khat, np.zeros(length), vhat, scale) for q in np.asarray(queries, dtype=np.float64)]
        return np.stack(outs), float(np.max(np.linalg.norm(vhat, axis=1)))
    block_size = cache["k_norm"].shape[2]
    rows = read_sequence(cache, table_row, length, kv_head, block_size)
    k_codes = packing.unpack_planes(rows["k_codes"], book["k_bits"], d)
    khat = reconstruct_mse(rows["k_norm"].reshape(-1), k_codes, book["rot"], book["k_levels"])
    vhat = reconstruct_mse(rows["v_norm"].reshape(-1), rows["v_code_values"], book["rot"], book["v_levels"])
    qjl = "k_qjl" in rows and book["proj"].shape[0] > 0
    signs = packing.unpack_signs(rows["k_qjl"], book["proj"].shape[0]) if qjl else None
    outs = []
    for query in np.asarray(queries, dtype=np.float64):
        corr = qjl_estimate(query, rows["k_rnorm"].reshape(-1), signs, book["proj"]) if qjl else np.zeros(length)
        outs.append(attend(query, khat, corr, vhat, scale))
    return np.stack(outs), float(np.max(np.linalg.norm(vhat, axis=1)))


def decode_attention(query, cache, table_row, length, kv_head, book, scale=None):
    """Output of one query head of one sequence, from the packed cache.

    ``book`` holds the oracle's own R, S, levels and bit widths:
    keys ``rot``, ``proj``, ``k_levels``, ``v_levels``, ``k_bits``, ``v_bits``.
    ``cache`` maps field names to arrays [num_blocks][n_kv][block_size][...]:
    ``k_codes``, ``k_qjl`` (may be absent when QJL is off), ``k_norm``,
    ``k_rnorm``, ``v_codes``, ``v_norm``.
    """
    d = book["rot"].shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if book.get("codec") == "polar":
        khat, vhat = _polar_rows(cache, table_row, length, kv_head, book)
        return attend(query, khat, np.zeros(length), vhat, scale), float(np.max(np.linalg.norm(vhat, axis=1)))
    block_size = cache["k_norm"].shape[2]
    rows = read_sequence(cache, table_row, length, kv_head, block_size)
    k_codes = packing.unpack_planes(rows["k_codes"], book["k_bits"], d)
    khat = reconstruct_mse(rows["k_norm"].reshape(-1), k_codes, book["rot"], book["k_levels"])
    if "k_qjl" in rows and book["proj"].shape[0] > 0:
        signs = packing.unpack_signs(rows["k_qjl"], book["proj"].shape[0])
        corr = qjl_estimate(query, rows["k_rnorm"].reshape(-1), signs, book["proj"])
    else:
        corr = np.zeros(length)
    v_codes = rows["v_code_values"]
    vhat = reconstruct_mse(rows["v_norm"].reshape(-1), v_codes, book["rot"], book["v_levels"])
    return attend(query, khat, corr, vhat, scale), float(np.max(np.linalg.norm(vhat, axis=1)))


def decode_attention_parts(query, parts, scale=None):
    """Output of one query head over a context split into parts, each read
    from its own cache with its own codebook (the yfxerp.com page, §2.3:
    prompt tokens kept at a higher bit width than generated ones): one
    softmax over the concatenation.  ``parts``: list of (cache, table_row,
    length, kv_head, book); the books share R and S.  Returns the output and
    max_t ||v_hat_t|| over every part."""
    khats, corrs, vhats = [], [], []
    d = parts[0][4]["rot"].shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for cache, table_row, length, kv_head, book in parts:
        if length == 0:
            continue
        rows = read_sequence(cache, table_row, length, kv_head, cache["k_norm"].shape[2])
        codes = packing.unpack_planes(rows["k_codes"], book["k_bits"], d)
        khats.append(reconstruct_mse(rows["k_norm"].reshape(-1), codes, book["rot"], book["k_levels"]))
        if "k_qjl" in rows and book["proj"].shape[0] > 0:
            signs = packing.unpack_signs(rows["k_qjl"], book["proj"].shape[0])
            corrs.append(qjl_estimate(query, rows["k_rnorm"].reshape(-1), signs, book["proj"]))
        else:
            corrs.append(np.zeros(length))
        vhats.append(reconstruct_mse(rows["v_norm"].reshape(-1), rows["v_code_values"], book["rot"],
                                     book["v_levels"]))
    if not khats:
        return np.zeros(d), 1.0
    khat, corr, vhat = np.concatenate(khats), np.concatenate(corrs), np.concatenate(vhats)
    return attend(query, khat, corr, vhat, scale), float(np.max(np.linalg.norm(vhat, axis=1)))
