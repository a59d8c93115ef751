"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than itself: published
test vectors, closed forms, independent quadrature, Monte Carlo, brute force,
or bounds printed on the pages (TurboQuant as summarised by the 甲子光年
article, §2 stage 1 / stage 2 and the distortion-rate paragraph at the end of
§2; intelliparadigm.com §2.1.1, §2.1.2, §2.2).
"""
import itertools
import math
import os

import numpy as np
import pytest
from scipy import integrate, special, stats

from oracle import attention, codebook, engine, packing, prng, quantize, rotation

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return [ln.strip() for ln in fh if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------- PRNG -----

def test_splitmix64_published_outputs():
    for line in _golden_lines("splitmix64.txt"):
        seed, outs = line.split(":")
        gen = prng.SplitMix64(int(seed))
        assert [gen.next_u64() for _ in outs.split()] == [int(v) for v in outs.split()]


def test_uniforms_in_open_closed_unit_interval_and_uniform():
    gen = prng.SplitMix64(99)
    u = np.array([gen.next_uniform() for _ in range(20000)])
    assert u.min() > 0.0 and u.max() <= 1.0
    assert stats.kstest(u, "uniform").pvalue > 1e-3


def test_box_muller_normals_are_standard_normal():
    z = np.array(prng.gaussians(5, 20001))
    assert len(z) == 20001
    assert stats.kstest(z, "norm").pvalue > 1e-3
    # cos/sin pairs of one radius are uncorrelated
    assert abs(np.corrcoef(z[0:-1:2], z[1::2])[0, 1]) < 0.05


# ------------------------------------------------------------ rotation -----

def test_rotation_is_orthogonal_to_1e12():
    rot, proj = rotation.rotation_and_projection(128, 128, 0)
    assert np.max(np.abs(rot.T @ rot - np.eye(128))) < 1e-12
    assert proj.shape == (128, 128)


def test_rotation_is_q_factor_with_positive_diagonal():
    gauss, _ = rotation.draw_matrices(64, 0, 3)
    rot = rotation.haar_from_gaussian(gauss)
    upper = rot.T @ gauss                      # = T, upper triangular
    assert np.max(np.abs(np.tril(upper, -1))) < 1e-10
    assert np.all(np.diag(upper) > 0)


def test_stream_order_g_then_s():
    values = prng.gaussians(11, 8 * 8 + 4 * 8)
    gauss, proj = rotation.draw_matrices(8, 4, 11)
    assert np.array_equal(gauss.ravel(), np.array(values[:64]))
    assert np.array_equal(proj.ravel(), np.array(values[64:]))


def test_haar_rotation_moves_a_fixed_vector_uniformly():
    # Haar law: R e1 is uniform on the sphere, so its coordinates follow f_d;
    # without the sign fix the first coordinate would be biased positive.
    d = 16
    rng = np.random.default_rng(0)
    first = np.array([rotation.haar_from_gaussian(rng.standard_normal((d, d)))[:, 0] for _ in range(3000)])
    assert stats.kstest(first[:, 0], lambda x: codebook.cdf(x, d)).pvalue > 1e-3
    assert stats.kstest(first[:, 5], lambda x: codebook.cdf(x, d)).pvalue > 1e-3
    assert abs(np.mean(first[:, 0])) < 4.0 / math.sqrt(d * 3000)


# ------------------------------------------------------- coordinate law -----

@pytest.mark.parametrize("d", [3, 8, 128, 1024])
def test_density_normalised_with_variance_one_over_d(d):
    mass, _ = integrate.quad(lambda x: float(codebook.density(x, d)), -1, 1, points=[0.0], limit=400)
    var, _ = integrate.quad(lambda x: x * x * float(codebook.density(x, d)), -1, 1, points=[0.0], limit=400)
    assert abs(mass - 1.0) < 1e-10
    assert abs(var - 1.0 / d) < 1e-10 / d


def test_cdf_matches_quadrature_and_first_moment_closed_form():
    d = 128
    for x in (-0.3, -0.05, 0.0, 0.02, 0.2):
        q, _ = integrate.quad(lambda u: float(codebook.density(u, d)), -1, x, points=[min(0.0, x)], limit=400)
        assert abs(float(codebook.cdf(x, d)) - q) < 1e-12
        m, _ = integrate.quad(lambda u: u * float(codebook.density(u, d)), -1, x, points=[min(0.0, x)], limit=400)
        assert abs(float(codebook.partial_first_moment(x, d)) - m) < 1e-13


def test_rotated_unit_vector_coordinates_follow_beta_law():
    # For a fixed vector (here spiky: one channel x40), the coordinates of
    # R x / ||x|| over Haar draws of R follow f_d, whatever x looks like.
    d = 128
    rng = np.random.default_rng(1)
    x = rng.standard_normal(d)
    x[3] *= 40.0
    x /= np.linalg.norm(x)
    y = np.array([rotation.haar_from_gaussian(rng.standard_normal((d, d))) @ x for _ in range(3000)])
    assert stats.kstest(y[:, 7], lambda t: codebook.cdf(t, d)).pvalue > 1e-3
    assert stats.kstest(y[:, 100], lambda t: codebook.cdf(t, d)).pvalue > 1e-3


# ------------------------------------------------------------ codebook -----

@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_lloyd_max_fixed_point_by_independent_quadrature(bits):
    d = 128
    levels, bounds = codebook.lloyd_max(d, bits)
    assert np.all(np.diff(levels) > 0)
    assert np.max(np.abs(bounds - 0.5 * (levels[:-1] + levels[1:]))) < 1e-15
    edges = np.concatenate(([-1.0], bounds, [1.0]))
    for i, level in enumerate(levels):
        pts = [0.0] if edges[i] < 0.0 < edges[i + 1] else None
        num, _ = integrate.quad(lambda x: x * float(codebook.density(x, d)), edges[i], edges[i + 1],
                                points=pts, epsabs=1e-18, epsrel=1e-13, limit=400)
        den, _ = integrate.quad(lambda x: float(codebook.density(x, d)), edges[i], edges[i + 1],
                                points=pts, epsabs=1e-18, epsrel=1e-13, limit=400)
        assert abs(num / den - level) < 1e-12
    # the coordinate law is even: the codebook is exactly odd-symmetric and the
    # middle boundary is exactly 0 (a coordinate at 0 takes the lower level)
    assert np.array_equal(levels, -levels[::-1])
    assert bounds[len(bounds) // 2] == 0.0
    assert np.searchsorted(bounds, 0.0, side="left") == len(levels) // 2 - 1


def test_one_bit_levels_closed_form():
    # 1-bit Lloyd-Max levels are +-E|X| = +-Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2)).
    for d in (8, 128):
        levels, bounds = codebook.lloyd_max(d, 1)
        expect = math.exp(math.lgamma(d / 2) - math.lgamma((d + 1) / 2)) / math.sqrt(math.pi)
        assert abs(levels[1] - expect) < 1e-14 and abs(levels[0] + expect) < 1e-14
        assert abs(bounds[0]) < 1e-15


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_high_dimension_limit_is_gaussian_lloyd_max(bits):
    table = {int(k): v for k, v in (ln.split(":") for ln in _golden_lines("gaussian_lloyd_max.txt"))}
    mse_txt, lv_txt = table[bits].split("|")
    published = np.array([float(v) for v in lv_txt.split()])
    d = 8192
    levels, bounds = codebook.lloyd_max(d, bits)
    scaled = levels[len(levels) // 2:] * math.sqrt(d)
    assert np.max(np.abs(scaled - published)) < 3e-3
    dist = codebook.mse_distortion(d, levels, bounds)
    assert abs(dist / float(mse_txt) - 1.0) < 2e-3


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_distortion_quadrature_matches_monte_carlo_and_page_bounds(bits):
    d = 128
    book = engine.build(d=d, k_bits=bits, v_bits=bits, qjl_m=0, seed=0)
    dist = codebook.mse_distortion(d, book["v_levels"], book["v_bounds"])
    # page bounds: >= 1/4^b for any quantizer, <= (sqrt(3) pi / 2) / 4^b for TurboQuant
    assert 4.0 ** -bits <= dist <= math.sqrt(3) * math.pi / 2 * 4.0 ** -bits
    rng = np.random.default_rng(bits)
    u = rng.standard_normal((20000, d))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    norm, _, codes = quantize.encode_mse(u, book["rot"], book["v_bounds"])
    err = np.sum((u - quantize.reconstruct_mse(norm, codes, book["rot"], book["v_levels"])) ** 2, axis=1)
    assert abs(np.mean(err) - dist) < 4 * np.std(err) / math.sqrt(len(err)) + 1e-6
    if bits == 1:
        levels = book["v_levels"]
        assert abs(dist - (1.0 - d * levels[1] ** 2)) < 1e-10
        assert abs(4 * dist - 1.45) < 0.02          # "about 1.45x" at b = 1


# ------------------------------------------------------ nearest level -----

@pytest.mark.parametrize("d,bits", [(8, 1), (4, 2), (6, 2)])
def test_per_coordinate_codes_equal_brute_force_codeword_search(d, bits):
    levels, bounds = codebook.lloyd_max(d, bits)
    codewords = np.array(list(itertools.product(levels, repeat=d)))
    index = np.array(list(itertools.product(range(len(levels)), repeat=d)))
    rng = np.random.default_rng(d * 10 + bits)
    y = rng.standard_normal((200, d))
    y /= np.linalg.norm(y, axis=1, keepdims=True)
    best = index[np.argmin(((y[:, None, :] - codewords[None]) ** 2).sum(-1), axis=1)]
    assert np.array_equal(quantize.nearest_level_codes(y, bounds), best)


def test_exhaustive_level_search_and_boundary_ties():
    levels, bounds = codebook.lloyd_max(128, 3)
    rng = np.random.default_rng(2)
    y = rng.normal(0, 0.12, 50000)
    assert np.array_equal(quantize.nearest_level_codes(y, bounds),
                          np.argmin(np.abs(y[:, None] - levels[None]), axis=1))
    # a coordinate exactly on a boundary takes the lower cell
    assert np.array_equal(quantize.nearest_level_codes(bounds, bounds), np.arange(len(bounds)))
    assert np.array_equal(quantize.nearest_level_codes(np.nextafter(bounds, 1), bounds), np.arange(len(bounds)) + 1)


def test_zero_vector_encoding():
    book = engine.build(k_bits=3, v_bits=2, qjl_m=128, seed=0)
    keys = engine.encode_keys(np.zeros((1, 128)), book)
    assert keys["k_norm"][0] == 0 and keys["k_rnorm"][0] == 0
    assert np.all(keys["codes"] == np.sum(book["k_bounds"] < 0))
    assert np.all(keys["signs"] == 0)


# -------------------------------------------------------------- packing -----

def test_packing_hand_worked_cases():
    for line in _golden_lines("packing.txt"):
        bits, codes, packed = (s.split() for s in line.split("|"))
        bits = int(bits[0])
        codes = np.array([[int(c) for c in codes]])
        expect = np.array([[int(b, 16) for b in packed]], dtype=np.uint8)
        assert np.array_equal(packing.pack_planes(codes, bits), expect)
        assert np.array_equal(packing.unpack_planes(expect, bits, codes.shape[1]), codes)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_packing_round_trip(bits):
    codes = np.random.default_rng(bits).integers(0, 1 << bits, size=(50, 128))
    packed = packing.pack_planes(codes, bits)
    assert packed.shape == (50, 16 * bits)
    assert np.array_equal(packing.unpack_planes(packed, bits, 128), codes)


def test_value_packing_hand_worked_case():
    field = np.zeros((1, 1, 2, 2, 1), dtype=np.uint8)
    codes = np.array([[(t + j) % 4 for j in range(2)] for t in range(8)])
    packing.write_value_codes(field, codes, np.arange(8), 0)
    for line in _golden_lines("value_packing.txt"):
        where, byte = line.split("|")
        p, j = (int(v) for v in where.split())
        assert field[0, 0, p, j, 0] == int(byte, 16)
    assert np.array_equal(packing.read_value_codes(field, np.arange(8), 0), codes)


def test_value_packing_round_trip_keeps_other_tokens_and_heads():
    rng = np.random.default_rng(8)
    field = rng.integers(0, 256, size=(3, 2, 3, 128, 8), dtype=np.uint8)
    before = field.copy()
    slots = np.array([5, 70, 191, 64])
    codes = rng.integers(0, 8, size=(4, 128))
    packing.write_value_codes(field, codes, slots, 1)
    assert np.array_equal(packing.read_value_codes(field, slots, 1), codes)
    assert np.array_equal(field[:, 0], before[:, 0])
    others = np.setdiff1d(np.arange(192), slots)
    assert np.array_equal(packing.read_value_codes(field, others, 1), packing.read_value_codes(before, others, 1))


def test_slot_index_layout():
    # [num_blocks][n_kv][block_size] rows: slot 70, head 1, 3 heads, 64-token blocks
    assert packing.slot_index(70, 1, 3, 64) == (1 * 3 + 1) * 64 + 6


# ---------------------------------------------------------------- QJL -----

def test_qjl_estimator_unbiased_with_predicted_variance():
    # E over S of gamma sqrt(pi/2)/m <S q, sign(S r)> = <q, r>  (10^4 draws of S)
    d = m = 128
    rng = np.random.default_rng(7)
    q = rng.standard_normal(d)
    r = 0.3 * q + rng.standard_normal(d)
    gamma = np.float32(np.linalg.norm(r))
    draws = []
    for _ in range(100):
        projs = rng.standard_normal((100, m, d))
        for proj in projs:
            signs = (proj @ r > 0).astype(np.int64)
            draws.append(attention.qjl_estimate(q, np.array([gamma]), signs[None], proj)[0])
    draws = np.array(draws)
    truth = float(q @ r) * float(gamma) / np.linalg.norm(r)
    var = (math.pi / 2 * (q @ q) * float(gamma) ** 2 - truth ** 2) / m
    assert abs(np.mean(draws) - truth) < 4 * math.sqrt(var / len(draws))
    assert abs(np.var(draws) / var - 1.0) < 0.06


def test_sign_convention_projected_greater_than_zero():
    book = engine.build(k_bits=2, v_bits=1, qjl_m=128, seed=1)
    x = np.random.default_rng(3).standard_normal((5, 128))
    norm, _, codes = quantize.encode_mse(x, book["rot"], book["k_bounds"])
    _, signs, z = quantize.encode_qjl(x, norm, codes, book["rot"], book["k_levels"], book["proj"])
    assert np.array_equal(signs, (z > 0).astype(np.int64))
    resid = x - quantize.reconstruct_mse(norm, codes, book["rot"], book["k_levels"])
    assert np.allclose(z, resid @ book["proj"].T)


def test_one_bit_mse_inner_product_bias_two_over_pi():
    # 1-bit stage-1 alone shrinks inner products: E_R <q, x_hat> = d c1^2 <q, x> -> 2/pi.
    d = 128
    levels, bounds = codebook.lloyd_max(d, 1)
    rng = np.random.default_rng(9)
    x = rng.standard_normal(d)
    x /= np.linalg.norm(x)
    q = 0.8 * x + 0.2 * rng.standard_normal(d)
    ratios = []
    for _ in range(2000):
        rot = rotation.haar_from_gaussian(rng.standard_normal((d, d)))
        norm, _, codes = quantize.encode_mse(x[None], rot, bounds)
        ratios.append(float(quantize.reconstruct_mse(norm, codes, rot, levels)[0] @ q) / float(q @ x))
    ratios = np.array(ratios)
    expect = d * levels[1] ** 2
    assert abs(np.mean(ratios) - expect) < 4 * np.std(ratios) / math.sqrt(len(ratios))
    assert abs(expect - 2 / math.pi) < 0.005


def test_full_key_estimator_unbiased_over_projections():
    # stage 1 + QJL: E_S[estimate] = <q, k> for fixed R and codes
    book = engine.build(k_bits=3, v_bits=2, qjl_m=128, seed=0)
    rng = np.random.default_rng(12)
    k = rng.standard_normal((1, 128)) * 3.0
    q = rng.standard_normal(128)
    norm, _, codes = quantize.encode_mse(k, book["rot"], book["k_bounds"])
    khat = quantize.reconstruct_mse(norm, codes, book["rot"], book["k_levels"])[0]
    est = []
    for _ in range(4000):
        proj = rng.standard_normal((128, 128))
        gamma, signs, _ = quantize.encode_qjl(k, norm, codes, book["rot"], book["k_levels"], proj)
        est.append(khat @ q + attention.qjl_estimate(q, gamma, signs, proj)[0])
    est = np.array(est)
    assert abs(np.mean(est) - float(k[0] @ q)) < 4 * np.std(est) / math.sqrt(len(est)) + 1e-4


# ------------------------------------------------------------ attention -----

def test_attention_reduces_to_textbook_softmax_without_quantization():
    rng = np.random.default_rng(4)
    q = rng.standard_normal(128)
    keys = rng.standard_normal((300, 128)) * 2
    vals = rng.standard_normal((300, 128))
    got = attention.attend(q, keys, np.zeros(300), vals, 1 / math.sqrt(128))
    expect = special.softmax(keys @ q / math.sqrt(128)) @ vals
    assert np.max(np.abs(got - expect)) < 1e-12


def test_attention_is_rotation_invariant():
    # attending in the rotated space then rotating back equals attending in
    # the original space (R^T R = I)
    rng = np.random.default_rng(5)
    rot, _ = rotation.rotation_and_projection(128, 0, 2)
    q = rng.standard_normal(128)
    keys = rng.standard_normal((64, 128))
    vals = rng.standard_normal((64, 128))
    plain = attention.attend(q, keys, np.zeros(64), vals, 0.1)
    rotated = attention.attend(rot @ q, keys @ rot.T, np.zeros(64), vals @ rot.T, 0.1) @ rot
    assert np.max(np.abs(plain - rotated)) < 1e-12


def test_cache_decode_uses_block_table_and_gqa_grouping():
    book = engine.build(k_bits=3, v_bits=3, qjl_m=128, seed=0)
    rng = np.random.default_rng(6)
    n_kv, bs = 2, 16
    k = rng.standard_normal((40, n_kv, 128))
    v = rng.standard_normal((40, n_kv, 128))
    cache = engine.empty_cache(book, 6, n_kv, bs)
    table = np.array([[4, 1, 5]])
    slots = table[0, np.arange(40) // bs] * bs + np.arange(40) % bs
    engine.append(cache, book, k, v, slots)
    q = rng.standard_normal((1, 4, 128))
    out, _ = engine.decode(q, cache, table, [40], book)
    # direct computation from the encoder outputs, head 3 -> kv head 1
    keys = engine.encode_keys(k[:, 1], book)
    vals = engine.encode_values(v[:, 1], book)
    khat = quantize.reconstruct_mse(keys["k_norm"], keys["codes"], book["rot"], book["k_levels"])
    vhat = quantize.reconstruct_mse(vals["v_norm"], vals["codes"], book["rot"], book["v_levels"])
    corr = attention.qjl_estimate(q[0, 3], keys["k_rnorm"], keys["signs"], book["proj"])
    expect = attention.attend(q[0, 3], khat, corr, vhat, 1 / math.sqrt(128))
    assert np.max(np.abs(out[0, 3] - expect)) < 1e-12


def test_group_decode_equals_per_head_decode():
    # decoding a GQA group's heads together reuses one reconstruction: same outputs
    from oracle import attention
    book = engine.build(k_bits=3, v_bits=2, qjl_m=128, seed=4)
    rng = np.random.default_rng(12)
    cache = engine.empty_cache(book, 2, 2, 64)
    k = rng.standard_normal((90, 2, 128))
    v = rng.standard_normal((90, 2, 128))
    engine.append(cache, book, k, v, np.arange(90))
    q = rng.standard_normal((3, 128))
    table = np.array([1, 0])
    outs, vmax = attention.decode_attention_heads(q, cache, table, 77, 1, book)
    for h in range(3):
        one, vm = attention.decode_attention(q[h], cache, table, 77, 1, book)
        assert np.array_equal(outs[h], one) and vm == vmax


def test_split_context_equals_one_cache():
    # a context split over two caches of one codebook attends exactly like the
    # same tokens in one cache (one softmax over the concatenation)
    from oracle import attention
    book = engine.build(k_bits=3, v_bits=3, qjl_m=128, seed=2)
    rng = np.random.default_rng(21)
    k = rng.standard_normal((150, 1, 128))
    v = rng.standard_normal((150, 1, 128))
    whole = engine.empty_cache(book, 3, 1, 64)
    engine.append(whole, book, k, v, np.arange(150))
    first = engine.empty_cache(book, 2, 1, 64)
    engine.append(first, book, k[:100], v[:100], np.arange(100))
    second = engine.empty_cache(book, 1, 1, 64)
    engine.append(second, book, k[100:], v[100:], np.arange(50))
    q = rng.standard_normal(128)
    ref, vmax = attention.decode_attention(q, whole, np.arange(3), 150, 0, book)
    got, vmax2 = attention.decode_attention_parts(q, [(first, np.arange(2), 100, 0, book),
                                                      (second, np.arange(1), 50, 0, book)])
    assert np.allclose(got, ref, rtol=0, atol=1e-12) and vmax == vmax2
