"""Device memory for the compressed cache and the decode workspace.

Torch provides the allocations; every computation is a library call.  Fields
are laid out as the ABI requires: [num_blocks][n_kv_heads][block_size][item].
"""
import torch

from . import binding


def allocate_cache(book, num_blocks, n_kv_heads, device="cuda"):
    """Dict of zero-filled device tensors, one per present cache field."""
    sizes = binding.tq_cache_field_bytes(book)
    bs = book.block_size
    cache = {}
    for name, nbytes in sizes.items():
        if nbytes == 0:
            continue
        if name == "v_codes" and getattr(book, "codec", 0) == binding.TQ_CODEC_POLAR:
            # PolarQuant records are token-major for values too
            cache[name] = torch.zeros((num_blocks, n_kv_heads, bs, nbytes), dtype=torch.uint8, device=device)
        elif name == "v_codes":
            # token-transposed inside a block: [block][head][plane][coordinate][block_size / 8]
            bits = nbytes * 8 // 128
            cache[name] = torch.zeros((num_blocks, n_kv_heads, bits, 128, bs // 8), dtype=torch.uint8, device=device)
        elif name.endswith("norm"):
            dt = torch.float16 if nbytes == 2 else torch.float32
            cache[name] = torch.zeros((num_blocks, n_kv_heads, bs), dtype=dt, device=device)
        else:
            cache[name] = torch.zeros((num_blocks, n_kv_heads, bs, nbytes), dtype=torch.uint8, device=device)
    return cache


def cache_view(book, cache):
    num_blocks, n_kv, bs = cache["k_norm"].shape
    return binding.make_cache_view(cache, num_blocks, n_kv, bs)


def allocate_workspace(book, batch, n_q_heads, max_context, device="cuda"):
    nbytes = binding.tq_decode_workspace_bytes(book, batch, n_q_heads, max_context)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device), nbytes


def cache_bytes_per_token_head(book):
    return sum(binding.tq_cache_field_bytes(book).values())
