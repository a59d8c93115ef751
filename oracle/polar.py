"""PolarQuant, the alternative stage 1 of the intelliparadigm.com page
(§2.1.1, step 2 "递归极坐标变换") -- test infrastructure only.

After the random rotation y = R x, the coordinates are taken in adjacent
pairs (y_0, y_1), (y_2, y_3), ...; each pair becomes a radius and an angle,
the angle is rounded to the nearest multiple of pi/12 (24 equal sectors of
the circle), and the radii are paired again the same way, level after level,
until a single radius -- the norm of the vector -- is left, which is kept.

Readings (the page prints the encoder only, with garbled bit counts):
* level 1 angles lie in (-pi, pi]; the code is the rounded multiple of pi/12
  taken modulo 24 (0..23, 5 bits).  From level 2 on both members of a pair
  are radii, so the angle lies in [0, pi/2] and the code in 0..6 (3 bits).
* angle = atan2(second member, first member); atan2(0, 0) = 0.
* rounding is half to even (the page rounds with Python's round).
* the radii of every level are those of the unquantized values; only the
  angles are quantized, so no decision depends on another.
* the decoder (not printed) inverts the recursion with the quantized angles:
  a radius r with angle code c becomes the pair (r cos(c pi/12), r sin(c pi/12)).
* the final radius is stored as float32; the reconstruction is R^T y_hat.
* record of d = 128 coordinates: the 64 level-1 codes x 5 bits, then the 63
  codes of levels 2..7 (32, 16, 8, 4, 2, 1 codes) x 3 bits, one little-endian
  bit stream (code i of a stream at bits [w i, w i + w), LSB first): 509 bits
  in 64 bytes.
* keys and values are both coded this way and carry no QJL bits; attention is
  the softmax of <q, x_hat_k> / sqrt(d) over the context, applied to x_hat_v.
"""
import math

import numpy as np

SECTOR = math.pi / 12.0
LEVEL1_CODES = 24
UPPER_CODES = 7          # angles in [0, pi/2]: codes 0..6
RECORD_BYTES = 64


def levels(d):
    """Number of pairing levels for a power-of-two dimension d."""
    n = int(round(math.log2(d)))
    if 1 << n != d:
        raise ValueError("d must be a power of two")
    return n


def _round_half_even(t):
    return np.rint(t).astype(np.int64)


def encode(y):
    """y [N, d] (rotated vectors, fp64) -> (codes: list of [N, d / 2^l] int
    arrays for levels l = 1..log2 d, radius [N] fp64, margins: list of [N, d / 2^l]
    distances of each pair's point to the nearest rounding boundary ray, in the
    units of y)."""
    cur = np.asarray(y, dtype=np.float64)
    codes, margins = [], []
    for lvl in range(1, levels(cur.shape[1]) + 1):
        first, second = cur[:, 0::2], cur[:, 1::2]
        theta = np.arctan2(second, first)
        rho = np.sqrt(first * first + second * second)
        t = theta / SECTOR
        k = _round_half_even(t)
        # the pair's distance to the ray at the rounding boundary nearest its angle
        boundary = (np.floor(t) + 0.5) * SECTOR
        margins.append(rho * np.abs(np.sin(theta - boundary)))
        codes.append(np.mod(k, LEVEL1_CODES) if lvl == 1 else k)
        cur = rho
    return codes, cur[:, 0], margins


def decode(codes, radius):
    """Inverse of ``encode`` with quantized angles: [N, d] fp64 rotated estimates."""
    cur = np.asarray(radius, dtype=np.float64)[:, None]
    for lvl_codes in reversed(codes):
        ang = np.asarray(lvl_codes, dtype=np.float64) * SECTOR
        nxt = np.empty((cur.shape[0], 2 * cur.shape[1]))
        nxt[:, 0::2] = cur * np.cos(ang)
        nxt[:, 1::2] = cur * np.sin(ang)
        cur = nxt
    return cur


def encode_vectors(x, rot):
    """x [N, d] -> (codes per level, radius stored as float32 [N], margins,
    y = R x fp64)."""
    x = np.asarray(x, dtype=np.float64)
    y = x @ np.asarray(rot, dtype=np.float64).T
    codes, radius, margins = encode(y)
    return codes, radius.astype(np.float32), margins, y


def reconstruct(codes, radius32, rot):
    """x_hat = R^T y_hat in the original space."""
    return decode(codes, radius32) @ np.asarray(rot, dtype=np.float64)


def _widths(d):
    return [5 if lvl == 1 else 3 for lvl in range(1, levels(d) + 1)]


def pack(codes):
    """Per-level codes -> [N, 64] uint8 records (d = 128)."""
    n = codes[0].shape[0]
    bits = []
    for lvl_codes, w in zip(codes, _widths(2 * codes[0].shape[1])):
        c = np.asarray(lvl_codes, dtype=np.int64)
        bits.append(((c[:, :, None] >> np.arange(w)) & 1).reshape(n, -1))
    stream = np.concatenate(bits, axis=1)
    out = np.zeros((n, RECORD_BYTES * 8), dtype=np.uint8)
    out[:, :stream.shape[1]] = stream
    return np.packbits(out, axis=1, bitorder="little")


def unpack(records, d=128):
    """[N, 64] uint8 records -> per-level codes."""
    stream = np.unpackbits(np.asarray(records, dtype=np.uint8), axis=1, bitorder="little").astype(np.int64)
    codes, pos = [], 0
    for lvl, w in enumerate(_widths(d), start=1):
        count = d >> lvl
        chunk = stream[:, pos:pos + count * w].reshape(-1, count, w)
        codes.append(np.sum(chunk << np.arange(w), axis=2))
        pos += count * w
    return codes
