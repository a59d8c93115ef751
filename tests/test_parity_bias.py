"""The inner-product bias of MSE-only keys against keys with the QJL bit, on
the GPU's own codes (甲子光年 article §2 第二階段: stage 1 alone shrinks inner
products -- by d c_1^2, near 2/pi, at 1 bit -- and the 1-bit QJL sketch of
the residual removes the shrinkage).  The estimates are decoded from the
GPU-written cache by the oracle; the expected slopes come from the codebook
(1 - D_mse for MSE-only keys, 1 with QJL)."""
import pytest

import bench

pytestmark = pytest.mark.gpu


def test_mse_only_keys_shrink_inner_products_and_qjl_removes_it():
    figs = bench._bias_figures(bench.bias_sample(n=4096, n_queries=16, seed=7))
    for f in figs:
        print(f)
        assert abs(f["slope"] - f["expected"]) <= 4.0 * f["stderr"] + 2e-3, f
    one_bit = [f for f in figs if f["k_bits"] == 1 and f["qjl_m"] == 0][0]
    assert 0.60 < one_bit["expected"] < 0.66          # d c_1^2 at d = 128 (2/pi ~ 0.637 as d grows)
    assert one_bit["slope"] < 0.7                      # and the GPU's codes show the shrinkage
    with_qjl = [f for f in figs if f["qjl_m"] > 0]
    assert all(abs(f["slope"] - 1.0) < 0.05 for f in with_qjl)
