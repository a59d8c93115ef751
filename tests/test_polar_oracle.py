"""Pins of the PolarQuant oracle (intelliparadigm.com page, §2.1.1 step 2)
against facts that do not come from the oracle itself: brute force over the
24 sectors, a product formula for the decoded coordinates, invariants of the
transform, the sector bound and a Monte Carlo check of the one-level error."""
import math

import numpy as np
import pytest

from oracle import engine, polar


def _wrap(a):
    return (a + math.pi) % (2.0 * math.pi) - math.pi


def test_one_pair_code_is_the_nearest_of_24_sectors():
    # brute force: the sector centre k pi/12 nearest to the point, found from
    # the complex argument of (a + ib) e^{-ik pi/12}
    rng = np.random.default_rng(1)
    pts = rng.standard_normal((2000, 2)) * rng.uniform(0.01, 10.0, size=(2000, 1))
    codes, radius, _ = polar.encode(pts)
    z = pts[:, 0] + 1j * pts[:, 1]
    ks = np.arange(24)
    dist = np.abs(np.angle(z[:, None] * np.exp(-1j * ks[None, :] * math.pi / 12.0)))
    assert np.array_equal(codes[0][:, 0], np.argmin(dist, axis=1))
    assert np.allclose(radius, np.abs(z), rtol=1e-14)
    # the decoded point is the sector centre at the same radius
    dec = polar.decode(codes, radius)
    cen = np.abs(z) * np.exp(1j * codes[0][:, 0] * math.pi / 12.0)
    assert np.allclose(dec[:, 0] + 1j * dec[:, 1], cen, atol=1e-12)


def _product_formula(level_codes, radius, d):
    # y_j = r * prod over levels l of cos or sin of the angle of j's ancestor
    # pair at level l (cos when bit l-1 of j is 0: the first member)
    out = np.empty((len(radius), d))
    for j in range(d):
        v = np.asarray(radius, dtype=np.float64).copy()
        for lvl, c in enumerate(level_codes, start=1):
            ang = c[:, j >> lvl] * math.pi / 12.0
            v = v * (np.sin(ang) if (j >> (lvl - 1)) & 1 else np.cos(ang))
        out[:, j] = v
    return out


@pytest.mark.parametrize("d", [8, 128])
def test_decoding_matches_the_product_formula_and_encoding_recovers_the_codes(d):
    rng = np.random.default_rng(d)
    n = 50
    nl = int(math.log2(d))
    # (upper-level code 0 gives its second member a zero radius, whose subtree
    # then has no angles to recover: codes 1..6 there)
    codes = [rng.integers(0, 24, size=(n, d >> 1))] + [rng.integers(1, 7, size=(n, d >> lvl))
                                                       for lvl in range(2, nl + 1)]
    radius = rng.uniform(0.5, 20.0, size=n)
    y = polar.decode(codes, radius)
    assert np.allclose(y, _product_formula(codes, radius, d), rtol=1e-12, atol=1e-12)
    back, r2, _ = polar.encode(y)
    assert np.allclose(r2, radius, rtol=1e-12)
    for lvl, (a, b) in enumerate(zip(codes, back), start=1):
        assert np.array_equal(a, b), lvl


def test_norms_are_kept_exactly():
    rng = np.random.default_rng(3)
    ref = engine.build(codec="polar")
    x = rng.standard_normal((200, 128)) * rng.uniform(0.1, 5.0, size=(200, 1))
    codes, radius32, _, y = polar.encode_vectors(x, ref["rot"])
    # the final radius is ||R x|| = ||x||, and every decoded vector has that norm
    assert np.allclose(radius32, np.linalg.norm(x, axis=1), rtol=2e-7)
    assert np.allclose(np.linalg.norm(polar.decode(codes, radius32), axis=1), radius32.astype(np.float64),
                       rtol=1e-12)


def test_every_angle_is_within_half_a_sector_and_codes_in_range():
    rng = np.random.default_rng(4)
    y = rng.standard_normal((300, 128))
    codes, radius, _ = polar.encode(y)
    cur = y
    for lvl, c in enumerate(codes, start=1):
        first, second = cur[:, 0::2], cur[:, 1::2]
        theta = np.arctan2(second, first)
        assert np.all(np.abs(_wrap(theta - c * math.pi / 12.0)) <= math.pi / 24.0 + 1e-12)
        if lvl == 1:
            assert c.min() >= 0 and c.max() <= 23
        else:
            assert c.min() >= 0 and c.max() <= 6
        cur = np.sqrt(first * first + second * second)


def test_one_level_error_matches_the_uniform_sector_closed_form():
    # a uniformly random direction in the plane is off its sector centre by an
    # angle uniform on [-pi/24, pi/24]: E|u - u_hat|^2 = 2 (1 - sinc) with
    # sinc = sin(pi/24) / (pi/24)
    rng = np.random.default_rng(5)
    ang = rng.uniform(-math.pi, math.pi, size=200000)
    pts = np.stack([np.cos(ang), np.sin(ang)], axis=1)
    codes, radius, _ = polar.encode(pts)
    err = np.sum((polar.decode(codes, radius) - pts) ** 2, axis=1)
    h = math.pi / 24.0
    expect = 2.0 * (1.0 - math.sin(h) / h)
    assert abs(err.mean() - expect) < 4.0 * err.std() / math.sqrt(err.size)


def test_margins_measure_the_distance_to_the_rounding_ray():
    # a point placed at a known angle off a sector boundary
    r, off = 3.0, 1e-3
    beta = 2.5 * math.pi / 12.0
    pts = np.array([[r * math.cos(beta + off), r * math.sin(beta + off)]])
    codes, _, margins = polar.encode(pts)
    assert codes[0][0, 0] == 3
    assert abs(margins[0][0, 0] - r * math.sin(off)) < 1e-12


def test_record_layout_by_hand():
    # level-1 code 0 = 1 -> bit 0; level-1 code 1 = 2 -> bit 6 (5 + 1);
    # level-2 code 0 = 5 (101b) -> bits 320 and 322; level-7 code = 6 (110b)
    # -> bits 320 + 3*62 + 1 and + 2 = 507, 508
    codes = [np.zeros((1, 128 >> lvl), dtype=np.int64) for lvl in range(1, 8)]
    codes[0][0, 0] = 1
    codes[0][0, 1] = 2
    codes[1][0, 0] = 5
    codes[6][0, 0] = 6
    rec = polar.pack(codes)
    assert rec.shape == (1, 64)
    bits = np.unpackbits(rec[0], bitorder="little")
    assert sorted(np.flatnonzero(bits).tolist()) == [0, 6, 320, 322, 507, 508]
    back = polar.unpack(rec)
    for a, b in zip(codes, back):
        assert np.array_equal(a, b)


def test_polar_cache_round_trip_and_attention_of_a_single_token():
    # a one-token context: softmax weight 1, the output is that token's
    # decoded value
    ref = engine.build(codec="polar", seed=2)
    rng = np.random.default_rng(6)
    k = rng.standard_normal((1, 1, 128))
    v = rng.standard_normal((1, 1, 128))
    cache = engine.empty_cache(ref, 1, 1, 64)
    keys, vals = engine.append(cache, ref, k, v, np.array([0]))
    out, vmax = engine.decode(rng.standard_normal((1, 1, 128)), cache, np.zeros((1, 1), dtype=np.int64),
                              np.array([1]), ref)
    vhat = polar.reconstruct(vals["codes"], vals["v_norm"], ref["rot"])[0]
    assert np.allclose(out[0, 0], vhat, atol=1e-12)
    assert abs(vmax[0, 0] - np.linalg.norm(vhat)) < 1e-12
