"""Lloyd-Max codebooks for one rotated coordinate (test infrastructure only).

甲子光年 article §2 第一階段: after a random rotation every coordinate of a
unit vector follows one known law (a Beta law, near-normal in high d, the
coordinates near-independent), so the MSE-optimal scalar quantizer for that
law -- the Lloyd-Max quantizer, a 1-D continuous k-means -- is computed once
per bit width, stored, and only looked up at inference.

Reading of "Beta分布": a coordinate x of a uniformly random unit vector in R^d
has (x + 1) / 2 ~ Beta((d-1)/2, (d-1)/2), i.e. density

    f_d(x) = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)) * (1 - x^2)^((d-3)/2)

on [-1, 1].  Lloyd-Max alternates the two optimality conditions: boundaries
are midpoints of neighbouring levels, levels are the centroids of their cells
under f_d.  The cell mass uses the regularised incomplete beta function
(scipy); the cell's first moment has the closed form

    int x (1 - x^2)^a dx = -(1 - x^2)^(a + 1) / (2 (a + 1)),  a = (d - 3) / 2.
"""
import math

import numpy as np
from scipy import integrate, special


def density_constant(d):
    """C_d = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)), via log-gamma."""
    return math.exp(math.lgamma(d / 2.0) - math.lgamma((d - 1) / 2.0)) / math.sqrt(math.pi)


def density(x, d):
    """f_d(x) for |x| <= 1 (zero outside)."""
    x = np.asarray(x, dtype=np.float64)
    inside = np.clip(1.0 - x * x, 0.0, None)
    return density_constant(d) * inside ** ((d - 3) / 2.0)


def cdf(x, d):
    """P(X <= x) = I_{(1+x)/2}((d-1)/2, (d-1)/2)."""
    p = (d - 1) / 2.0
    return special.betainc(p, p, np.clip((1.0 + np.asarray(x, dtype=np.float64)) / 2.0, 0.0, 1.0))


def survival(x, d):
    """P(X > x) = P(X < -x) by symmetry; accurate in the upper tail."""
    return cdf(-np.asarray(x, dtype=np.float64), d)


def cell_masses(edges, d):
    """P(edges[i] < X <= edges[i+1]) for every cell, each taken from the tail
    nearer the cell so that far-tail cells suffer no cancellation."""
    edges = np.asarray(edges, dtype=np.float64)
    lo, hi = edges[:-1], edges[1:]
    lower = cdf(hi, d) - cdf(lo, d)
    upper = survival(lo, d) - survival(hi, d)
    return np.where(lo >= 0.0, upper, lower)


def partial_first_moment(x, d):
    """int_{-1}^{x} u f_d(u) du = -C_d (1 - x^2)^(a+1) / (2 (a+1))."""
    a1 = (d - 1) / 2.0
    x = np.asarray(x, dtype=np.float64)
    return -density_constant(d) * np.clip(1.0 - x * x, 0.0, None) ** a1 / (2.0 * a1)


def centroids(edges, d):
    """E[X | edges[i] < X <= edges[i+1]] for every cell."""
    moment = partial_first_moment(edges, d)
    return (moment[1:] - moment[:-1]) / cell_masses(edges, d)


def lloyd_max(d, bits, tol=1e-13, max_iter=100000):
    """(levels, boundaries) of the 2^bits-level Lloyd-Max quantizer for f_d.

    Levels ascend; boundaries[i] separates levels i and i+1.  The start is the
    set of quantile midpoints; iteration stops once no level moves by more than
    ``tol`` in the sqrt(d)-scaled coordinate (fp64 rounding keeps the step
    near 1e-14 there, so the default stops just above that floor).
    """
    count = 1 << bits
    p = (d - 1) / 2.0
    probs = (np.arange(count) + 0.5) / count
    levels = 2.0 * special.betaincinv(p, p, probs) - 1.0
    scale = math.sqrt(d)
    for _ in range(max_iter):
        bounds = 0.5 * (levels[:-1] + levels[1:])
        new = centroids(np.concatenate(([-1.0], bounds, [1.0])), d)
        moved = np.max(np.abs(new - levels)) * scale
        levels = new
        if moved < tol:
            break
    # f_d is even, so the exact fixed point is odd-symmetric (c_i = -c_{K-1-i})
    # and its middle boundary is exactly 0; rounding in the iteration leaves a
    # residue near 1e-16 there, which would decide the tie at y = 0 (reading:
    # a tie goes to the lower level) by noise.  Restore the symmetry.
    levels = 0.5 * (levels - levels[::-1])
    bounds = 0.5 * (levels[:-1] + levels[1:])
    return levels, bounds


def mse_distortion(d, levels, bounds):
    """d * E[(X - Q(X))^2] for one coordinate: the expected ||u - u_hat||^2 of
    a unit vector quantized coordinate-wise (numerical quadrature per cell)."""
    edges = np.concatenate(([-1.0], np.asarray(bounds, dtype=np.float64), [1.0]))
    total = 0.0
    for i, level in enumerate(levels):
        val, _ = integrate.quad(lambda x: (x - level) ** 2 * float(density(x, d)),
                                edges[i], edges[i + 1], epsabs=1e-16, epsrel=1e-12, limit=200)
        total += val
    return d * total
