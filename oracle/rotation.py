"""Seeded Haar rotation R and Gaussian QJL matrix S (test infrastructure only).

* R: 甲子光年 article §2 第一階段 (a random rotation applied before the
  scalar quantizer) and intelliparadigm.com §2.1.1 step 1 (the orthogonal
  matrix is drawn from the Haar law).  A Haar-distributed orthogonal matrix is
  the Q factor of a d x d standard Gaussian matrix G = Q T once the signs are
  fixed so that diag(T) > 0 (Mezzadri, "How to generate random matrices from
  the classical compact groups", Notices AMS 2007).  The QR is numpy's
  (LAPACK Householder); the sign fix is applied here.
* S: m x d with i.i.d. N(0, 1) entries, the random projection of QJL
  (intelliparadigm.com §2.1.2; 甲子光年 §2 第二階段).

Stream order (a reading; the pages fix none): one SplitMix64/Box-Muller
stream seeded with ``seed``; the first d*d normals fill G row-major, the next
m*d fill S row-major.
"""
import numpy as np

from . import prng


def draw_matrices(d, m, seed):
    """Return (G, S) as float64 arrays from one seeded stream."""
    values = prng.gaussians(seed, d * d + m * d)
    gauss = np.array(values[: d * d], dtype=np.float64).reshape(d, d)
    proj = np.array(values[d * d:], dtype=np.float64).reshape(m, d) if m else np.zeros((0, d))
    return gauss, proj


def haar_from_gaussian(gauss):
    """Q of G = Q T with the column signs chosen so that diag(T) > 0."""
    q, t = np.linalg.qr(gauss)
    signs = np.sign(np.diag(t))
    signs[signs == 0] = 1.0
    return q * signs[None, :]


def rotation_and_projection(d, m, seed):
    """(R, S): the rotation y = R x and the QJL projection z = S r."""
    gauss, proj = draw_matrices(d, m, seed)
    return haar_from_gaussian(gauss), proj
