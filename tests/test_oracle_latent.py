"""Pins of the oracle's SpecFLASH latent compressor, softmax(Q . F^T) . F.

Fixed by closed forms (all features equal -> that feature; zero queries ->
the mean feature; queries scaled up -> the feature with the largest score),
a two-feature hand example, invariance to the order of the features, and the
library's scaled-dot-product attention in fp64 with scale 1.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def test_equal_features_give_that_feature():
    rng = np.random.default_rng(0)
    f = np.tile(rng.standard_normal(24), (9, 1))
    q = rng.standard_normal((5, 24))
    out = oracle.latent_compress(q, f)
    assert np.allclose(out, np.tile(f[0], (5, 1)), rtol=0, atol=1e-13)


def test_zero_queries_give_the_mean_feature():
    rng = np.random.default_rng(1)
    f = rng.standard_normal((37, 16))
    out = oracle.latent_compress(np.zeros((3, 16)), f)
    assert np.allclose(out, np.tile(f.mean(0), (3, 1)), rtol=0, atol=1e-13)


def test_large_queries_select_the_best_feature():
    rng = np.random.default_rng(2)
    f = rng.standard_normal((50, 8))
    q = rng.standard_normal((4, 8))
    best = (q @ f.T).argmax(1)
    gap = np.sort(q @ f.T, axis=1)
    lam = 60.0 / (gap[:, -1] - gap[:, -2]).min()   # every runner-up below e^-60
    out = oracle.latent_compress(q * lam, f)
    assert np.allclose(out, f[best], rtol=0, atol=1e-20 + 1e-12)


def test_two_features_by_hand():
    # scores 0 and ln 3 -> weights 1/4 and 3/4
    out = oracle.latent_compress(np.array([[1.0]]), np.array([[0.0], [math.log(3.0)]]))
    assert out.shape == (1, 1) and abs(out[0, 0] - 0.75 * math.log(3.0)) < 1e-15


def test_feature_order_does_not_matter():
    rng = np.random.default_rng(3)
    f = rng.standard_normal((2, 64, 12))
    q = rng.standard_normal((6, 12)) * 0.5
    perm = rng.permutation(64)
    a = oracle.latent_compress(q, f)
    b = oracle.latent_compress(q, f[:, perm])
    assert a.shape == (2, 6, 12) and np.allclose(a, b, rtol=0, atol=1e-13)


@pytest.mark.parametrize("Cq,N,d", [(64, 576, 32), (36, 324, 48), (1, 1, 5)])
def test_equals_library_attention_with_scale_one(Cq, N, d):
    rng = np.random.default_rng(Cq + N)
    f = rng.standard_normal((3, N, d))
    q = rng.standard_normal((Cq, d)) / math.sqrt(d)
    out = oracle.latent_compress(q, f)
    ft = torch.from_numpy(f)
    qt = torch.from_numpy(q).expand(3, Cq, d)
    want = torch.nn.functional.scaled_dot_product_attention(qt, ft, ft, scale=1.0).numpy()
    assert np.allclose(out, want, rtol=0, atol=1e-12)


def test_separate_values_follow_the_library_too():
    rng = np.random.default_rng(9)
    f = rng.standard_normal((40, 10))
    v = rng.standard_normal((40, 10))
    q = rng.standard_normal((7, 10)) * 0.3
    out = oracle.latent_compress(q, f, v)
    want = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(f)[None], torch.from_numpy(v)[None], scale=1.0)[0].numpy()
    assert np.allclose(out, want, rtol=0, atol=1e-12)
