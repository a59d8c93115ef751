"""Seeded synthetic inputs for tests and the benchmark (no method arithmetic).

The pages measure on LLM KV caches (Llama-3-8B / 70B, Gemma); no model
weights or datasets exist here, so K/V/query tensors are drawn with the
shapes and value structure of those workloads: standard normals, per-(head,
channel) scale profiles and a few outlier channels -- the energy spikes the
random rotation is meant to spread (seo-farm page §2 "旋转变换预处理").

Bulk tensors come from a seeded torch.Generator on the target device; small
choices (channel scales, outlier channels, context lengths, block
permutations) from numpy's default_rng.  This module is shared by the oracle
tests and the CUDA-path tests/bench; it contains nothing of the codec.
"""
import math

import numpy as np
import torch

HEAD_DIM = 128

# Workload configurations (sizes follow the benchmark's configuration list).
CONFIGS = {
    "c1_single_head_parity": dict(
        batch=1, n_q=1, n_kv=1, context=4096, dtype="fp32", k_bits=3, v_bits=3, qjl_m=128,
        block_size=64, log_uniform=None, outliers=4, outlier_scale=20.0, seed=0),
    "c2_llama3_8b_decode": dict(
        batch=16, n_q=32, n_kv=8, context=8192, dtype="bf16", k_bits=3, v_bits=3, qjl_m=128,
        block_size=64, log_uniform=(0.1, 10.0), outliers=3, outlier_scale=30.0, seed=0),
    "c3_prefill_quantize": dict(
        tokens=32768, n_kv=8, dtype="bf16", bit_sweep=(2, 3, 4), qjl_m=128, block_size=64,
        student_t_channels=3, seed=0),
    "c4_long_context": dict(
        batch=1, n_q=64, n_kv=8, context=131072, dtype="bf16", k_bits=4, v_bits=2, qjl_m=128,
        block_size=64, log_uniform=None, outliers=1, outlier_scale=50.0, seed=0),
    "c5_llama3_70b_paged": dict(
        batch=64, n_q=64, n_kv=8, context=(1024, 32768), dtype="bf16", k_bits=3, v_bits=3, qjl_m=128,
        block_size=64, log_uniform=(0.1, 10.0), outliers=0, outlier_scale=1.0, shuffled_table=True, seed=0),
}
# the same paged decode with 16-bit stored norms (102 bytes per token-head)
CONFIGS["c5_llama3_70b_paged_fp16_norms"] = dict(CONFIGS["c5_llama3_70b_paged"], norm_bits=16)
# the 8B-shaped decode over a PolarQuant cache (codec 1: 64-byte records, float32 radii, no QJL)
CONFIGS["c2_llama3_8b_decode_polar"] = dict(CONFIGS["c2_llama3_8b_decode"], codec=1, k_bits=0, v_bits=0, qjl_m=0)


def torch_dtype(name):
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def channel_scales(seed, n_kv, log_uniform=None, outliers=0, outlier_scale=1.0, d=HEAD_DIM):
    """[n_kv][d] multiplicative profile: log-uniform per (head, channel) if
    given, times ``outlier_scale`` on ``outliers`` seeded channels per head."""
    rng = np.random.default_rng(seed)
    if log_uniform is None:
        scales = np.ones((n_kv, d))
    else:
        lo, hi = log_uniform
        scales = np.exp(rng.uniform(math.log(lo), math.log(hi), size=(n_kv, d)))
    for h in range(n_kv):
        if outliers:
            scales[h, rng.choice(d, size=outliers, replace=False)] *= outlier_scale
    return scales


def gaussian_tokens(n_tokens, scales, dtype, device, generator):
    """[n_tokens][n_kv][d] = N(0, 1) * scales, cast to ``dtype``."""
    n_kv, d = scales.shape
    x = torch.randn((n_tokens, n_kv, d), generator=generator, device=device, dtype=torch.float32)
    x *= torch.as_tensor(scales, dtype=torch.float32, device=device)
    return x.to(dtype)


def student_t_tokens(n_tokens, n_kv, heavy_channels, dtype, device, generator, seed, d=HEAD_DIM):
    """N(0, 1) tokens whose ``heavy_channels`` seeded channels per head hold
    Student-t(3) samples instead (normal / sqrt(chi^2_3 / 3))."""
    x = torch.randn((n_tokens, n_kv, d), generator=generator, device=device, dtype=torch.float32)
    rng = np.random.default_rng(seed + 7)
    for h in range(n_kv):
        chans = torch.as_tensor(rng.choice(d, size=heavy_channels, replace=False), device=device)
        z = torch.randn((n_tokens, heavy_channels), generator=generator, device=device)
        chi = torch.randn((n_tokens, heavy_channels, 3), generator=generator, device=device).pow(2).sum(-1)
        x[:, h, chans] = z / torch.sqrt(chi / 3.0)
    return x.to(dtype)


def queries(batch, n_q, dtype, device, generator, d=HEAD_DIM):
    return torch.randn((batch, n_q, d), generator=generator, device=device, dtype=torch.float32).to(dtype)


def context_lengths(cfg, seed):
    ctx = cfg["context"]
    if isinstance(ctx, tuple):
        rng = np.random.default_rng(seed + 11)
        return rng.integers(ctx[0], ctx[1], endpoint=True, size=cfg["batch"]).astype(np.int32)
    return np.full(cfg["batch"], ctx, dtype=np.int32)


def block_layout(context_lens, block_size, shuffled, seed):
    """(block_table [batch][max_blocks] int32, num_blocks): every sequence gets
    ceil(ctx / block_size) blocks; physical ids are a seeded permutation of all
    blocks when ``shuffled`` (unused table entries are -1)."""
    need = [(int(c) + block_size - 1) // block_size for c in context_lens]
    max_blocks = max(1, max(need))
    num_blocks = max(1, sum(need))
    ids = np.arange(num_blocks, dtype=np.int32)
    if shuffled:
        ids = np.random.default_rng(seed + 13).permutation(num_blocks).astype(np.int32)
    table = np.full((len(need), max_blocks), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(need):
        table[b, :n] = ids[pos:pos + n]
        pos += n
    return table, num_blocks


def slots_for(block_table_row, positions, block_size):
    """Cache slots (physical block * block_size + offset) of token positions."""
    positions = np.asarray(positions, dtype=np.int64)
    return block_table_row[positions // block_size].astype(np.int64) * block_size + positions % block_size


def bf16_round_numpy(x):
    """float64 array rounded to the nearest bfloat16 (ties to even), as float64:
    the values a bf16 input tensor holds, for host-side (oracle) workloads."""
    bits = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)
