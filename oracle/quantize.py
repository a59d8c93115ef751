"""TurboQuant encoder for one head vector (test infrastructure only).

Stage 1, 甲子光年 article §2 第一階段: keep the norm, rotate the unit vector
with R, and replace every rotated coordinate by the nearest Lloyd-Max level
(the cell index is the code).  Stage 2, §2 第二階段: with a total budget of
b bits, keys use b-1 bits for stage 1 and one more bit per projected
coordinate for QJL on the residual (the difference between the vector and its
stage-1 reconstruction), keeping the residual norm; intelliparadigm.com §2.1.2
gives the sketch as ``projection_matrix @ residual > 0``.

Readings: the norm is stored as float32 and the reconstruction that defines
the residual uses that stored value; a coordinate exactly on a boundary takes
the lower cell; the zero vector gets y = 0 (codes of the cell holding 0),
residual 0, norm 0 and all sign bits 0.
"""
import numpy as np


def nearest_level_codes(y, bounds):
    """code_j = #{i : bounds[i] < y_j}: the nearest level of an ascending
    Lloyd-Max codebook whose boundaries are the level midpoints."""
    return np.searchsorted(np.asarray(bounds, dtype=np.float64), y, side="left")


def encode_mse(x, rot, bounds, norm_dtype=np.float32):
    """x [N, d] -> (stored norm [N] in norm_dtype -- float32, or float16 for a
    cache with 16-bit norms --, y [N, d] fp64 unit rotated vectors, codes [N, d])."""
    x = np.asarray(x, dtype=np.float64)
    norm = np.sqrt(np.sum(x * x, axis=1))
    safe = np.where(norm > 0.0, norm, 1.0)
    y = (x @ rot.T) / safe[:, None]
    y[norm == 0.0] = 0.0
    return norm.astype(norm_dtype), y, nearest_level_codes(y, bounds)


def reconstruct_mse(norm32, codes, rot, levels):
    """Stage-1 reconstruction in the original space: ||x|| R^T c[code]."""
    lv = np.asarray(levels, dtype=np.float64)[np.asarray(codes)]
    return norm32.astype(np.float64)[:, None] * (lv @ rot)


def encode_qjl(x, norm32, codes, rot, levels, proj, norm_dtype=np.float32):
    """Residual sketch against the stored norm ``norm32`` (float32 or float16):
    (gamma [N] in norm_dtype, signs [N, m] 0/1, z = S r [N, m] fp64)."""
    x = np.asarray(x, dtype=np.float64)
    resid = x - reconstruct_mse(norm32, codes, rot, levels)
    gamma = np.sqrt(np.sum(resid * resid, axis=1))
    z = resid @ np.asarray(proj, dtype=np.float64).T
    return gamma.astype(norm_dtype), (z > 0.0).astype(np.int64), z


def boundary_distance(y, bounds):
    """min_i |y_j - bounds[i]| per coordinate (unit-vector coordinates)."""
    b = np.asarray(bounds, dtype=np.float64)
    return np.min(np.abs(np.asarray(y)[..., None] - b), axis=-1)
