"""Bit layout of the compressed cache (test infrastructure only).

The pages fix what is stored -- b-bit codebook indices with no scale or
zero-point (甲子光年 §2 第一階段), the QJL sign bits of the residual plus its
norm (§2 第二階段) -- but not the byte layout.  Readings taken:

* Codes of one d-vector at beta bits are stored as beta bit-planes of d bits:
  plane p holds bit p of every code; within a plane, coordinate j is bit
  (j mod 8) of byte (j div 8) (least significant bit first).  A vector takes
  beta * d / 8 bytes, 16 * beta at d = 128, so every plane is 16-byte aligned.
* QJL signs: bit k (LSB first in byte k div 8) is 1 exactly when the k-th
  projected residual is > 0 (intelliparadigm.com §2.1.2 keeps
  ``projected > 0``).
* Paging: slot s lives in block s div block_size at offset s mod block_size.
  Key fields and all norms are arrays [num_blocks][n_kv_heads][block_size][item]
  (one row per token).
* Value codes are stored token-transposed inside a block (a reading chosen so
  that decode can contract over tokens): the value field is
  [num_blocks][n_kv_heads][bits][d][block_size / 8]; for plane p and
  coordinate j, bit (t mod 8) of byte (t div 8) holds bit p of the code of the
  token at offset t.  Per block and head this is the same bits * d *
  block_size / 8 bytes as the token-major form.
"""
import numpy as np


def pack_planes(codes, bits):
    """codes [N, d] (ints < 2^bits) -> uint8 [N, bits * d / 8]."""
    codes = np.asarray(codes, dtype=np.int64)
    n, d = codes.shape
    out = np.zeros((n, bits, d // 8), dtype=np.uint8)
    for p in range(bits):
        plane = (codes >> p) & 1
        for j in range(d):
            out[:, p, j // 8] |= (plane[:, j] << (j % 8)).astype(np.uint8)
    return out.reshape(n, bits * d // 8)


def unpack_planes(packed, bits, d):
    """uint8 [N, bits * d / 8] -> codes [N, d]."""
    packed = np.asarray(packed, dtype=np.uint8).reshape(-1, bits, d // 8)
    codes = np.zeros((packed.shape[0], d), dtype=np.int64)
    for p in range(bits):
        for j in range(d):
            bit = (packed[:, p, j // 8] >> (j % 8)) & 1
            codes[:, j] |= bit.astype(np.int64) << p
    return codes


def pack_signs(signs):
    """0/1 array [N, m] -> uint8 [N, m / 8]."""
    return pack_planes(np.asarray(signs, dtype=np.int64), 1)


def unpack_signs(packed, m):
    """uint8 [N, m / 8] -> 0/1 array [N, m]."""
    return unpack_planes(packed, 1, m)


def slot_index(slot, head, n_kv_heads, block_size):
    """Row of (slot, head) in a field array flattened to [-1, bytes_per_item]."""
    slot = np.asarray(slot, dtype=np.int64)
    block = slot // block_size
    offset = slot % block_size
    return (block * n_kv_heads + head) * block_size + offset


def write_value_codes(field, codes, slots, head):
    """Store codes [N, d] of tokens at ``slots`` (one KV head) into a value
    field [num_blocks][n_kv][bits][d][block_size / 8] (uint8, in place)."""
    bits, d, nbytes = field.shape[2], field.shape[3], field.shape[4]
    block_size = nbytes * 8
    codes = np.asarray(codes, dtype=np.int64)
    for n, slot in enumerate(np.asarray(slots, dtype=np.int64)):
        block, off = int(slot) // block_size, int(slot) % block_size
        for p in range(bits):
            for j in range(d):
                byte = field[block, head, p, j, off // 8]
                bit = (int(codes[n, j]) >> p) & 1
                byte = (int(byte) & ~(1 << (off % 8))) | (bit << (off % 8))
                field[block, head, p, j, off // 8] = byte


def read_value_codes(field, slots, head):
    """Codes [N, d] of the tokens at ``slots`` (one KV head) from a value field."""
    bits, d, nbytes = field.shape[2], field.shape[3], field.shape[4]
    block_size = nbytes * 8
    slots = np.asarray(slots, dtype=np.int64)
    block, off = slots // block_size, slots % block_size
    codes = np.zeros((len(slots), d), dtype=np.int64)
    for p in range(bits):
        for j in range(d):
            byte = field[block, head, p, j, off // 8].astype(np.int64)
            codes[:, j] |= ((byte >> (off % 8)) & 1) << p
    return codes
