"""Pins of the oracle's Sequential Temperature Scaling fit (one inverse
temperature per block position, minimising the BCE of sigmoid(beta z)
against the accept labels).  The pages name the calibration without a
formula, so these pins tie the oracle to temperature scaling's definition:
a library minimiser of the library BCE, a closed form and invariances."""
import numpy as np
import pytest
import torch

N, GAMMA = 4000, 5


def _logits(seed, scale=2.0):
    return np.random.default_rng(seed).normal(0, scale, (N, GAMMA)).astype(np.float32)


def test_sts_soft_labels_give_back_the_temperature(oracle):
    """Labels sigmoid(z / T_k) are matched exactly at beta_k = 1 / T_k."""
    z = _logits(1)
    T = np.array([0.25, 0.5, 1.0, 2.0, 7.0])
    a = (1.0 / (1.0 + np.exp(-z.astype(np.float64) / T))).astype(np.float32)
    res = oracle.sts_fit(z, a)
    assert np.all(res["status"] == 0)
    np.testing.assert_allclose(res["beta"], 1.0 / T, rtol=1e-5)


def test_sts_agrees_with_a_library_minimiser(oracle):
    """Hard Bernoulli labels from a miscalibrated confidence: beta_k is the
    minimiser of the library BCE-with-logits (scipy bounded scalar search)."""
    from scipy.optimize import minimize_scalar
    rng = np.random.default_rng(2)
    z = _logits(2)
    true_T = np.array([0.6, 1.0, 1.7, 3.0, 1.2])
    a = (rng.random((N, GAMMA)) < 1.0 / (1.0 + np.exp(-z / true_T))).astype(np.float32)
    res = oracle.sts_fit(z, a)
    for k in range(GAMMA):
        zk = torch.from_numpy(z[:, k].astype(np.float64))
        ak = torch.from_numpy(a[:, k].astype(np.float64))
        f = lambda b: float(torch.nn.functional.binary_cross_entropy_with_logits(b * zk, ak, reduction="sum"))
        m = minimize_scalar(f, bounds=(0.0, 20.0), method="bounded", options=dict(xatol=1e-10))
        assert res["status"][k] == 0
        np.testing.assert_allclose(res["beta"][k], m.x, rtol=1e-6)
        # and the fit sits near the generating temperature
        assert abs(res["beta"][k] * true_T[k] - 1.0) < 0.15


def test_sts_scale_invariance(oracle):
    """Scaling every logit by c divides beta by c."""
    rng = np.random.default_rng(3)
    z = _logits(3)
    a = rng.random((N, GAMMA)).astype(np.float32)
    a = np.where(z > 0, np.maximum(a, 0.3), np.minimum(a, 0.7)).astype(np.float32)
    b1 = oracle.sts_fit(z, a)["beta"]
    b4 = oracle.sts_fit((z * 4.0).astype(np.float32), a)["beta"]  # exact in fp32
    np.testing.assert_allclose(b4, b1 / 4.0, rtol=1e-9)


def test_sts_mask(oracle):
    """Masked pairs do not count: garbage in them changes nothing."""
    rng = np.random.default_rng(4)
    z = _logits(4)
    a = (rng.random((N, GAMMA)) < 1.0 / (1.0 + np.exp(-z))).astype(np.float32)
    mask = (rng.random((N, GAMMA)) < 0.7).astype(np.uint8)
    a2 = np.where(mask == 1, a, 1.0 - a).astype(np.float32)
    r1 = oracle.sts_fit(z, a, mask)
    r2 = oracle.sts_fit(z, a2, mask)
    np.testing.assert_array_equal(r1["beta"], r2["beta"])
    for k in range(GAMMA):  # the fit of position k on its kept pairs alone
        keep = mask[:, k] == 1
        one = oracle.sts_fit(z[keep, k:k + 1].copy(), a[keep, k:k + 1].copy())
        np.testing.assert_allclose(r1["beta"][k], one["beta"][0], rtol=1e-12)


def test_sts_degenerate_positions(oracle):
    """No information -> beta 1 (status 1); labels separated by the sign of z
    -> the cap 2^20 (status 2); labels against the sign of z -> beta 0."""
    z = _logits(5)
    a = np.random.default_rng(5).random((N, GAMMA)).astype(np.float32)
    a[:, 4] = 1.0 / (1.0 + np.exp(-z[:, 4]))  # calibrated: beta near 1
    z[:, 0] = 0.0
    a[:, 1] = (z[:, 1] > 0).astype(np.float32)
    a[:, 2] = (z[:, 2] < 0).astype(np.float32)
    mask = np.ones((N, GAMMA), np.uint8)
    mask[:, 3] = 0
    res = oracle.sts_fit(z, a, mask)
    assert res["status"].tolist()[:4] == [1, 2, 0, 1]
    assert res["beta"][0] == 1.0 and res["beta"][1] == 2.0 ** 20 and res["beta"][2] == 0.0 and res["beta"][3] == 1.0
    assert res["status"][4] == 0 and abs(res["beta"][4] - 1.0) < 1e-5


def test_sts_nearly_separated_labels_have_a_finite_fit(oracle):
    """a = sigmoid(z) above zero and a = 0 below: every label agrees in sign
    with z but the positive side is soft, so the minimiser is finite (and
    the library minimiser finds the same point)."""
    from scipy.optimize import minimize_scalar
    z = _logits(6)[:, :1].copy()
    a = np.where(z > 0, 1.0 / (1.0 + np.exp(-z)), 0.0).astype(np.float32)
    res = oracle.sts_fit(z, a)
    assert res["status"][0] == 0 and 0 < res["beta"][0] < 2.0 ** 20
    zk, ak = torch.from_numpy(z[:, 0].astype(np.float64)), torch.from_numpy(a[:, 0].astype(np.float64))
    f = lambda b: float(torch.nn.functional.binary_cross_entropy_with_logits(b * zk, ak, reduction="sum"))
    m = minimize_scalar(f, bounds=(0.0, 50.0), method="bounded", options=dict(xatol=1e-10))
    np.testing.assert_allclose(res["beta"][0], m.x, rtol=1e-6)


def test_sts_invalid_pairs(oracle):
    """A non-finite logit or a label outside [0, 1] in a counted pair fails
    its position (status 3, beta NaN); the same pair masked out does not."""
    z = _logits(7)
    a = (1.0 / (1.0 + np.exp(-z))).astype(np.float32)
    z[10, 0] = np.nan
    z[11, 1] = np.inf
    a[12, 2] = 1.5
    a[13, 3] = np.nan
    res = oracle.sts_fit(z, a)
    assert res["status"].tolist() == [3, 3, 3, 3, 0] and np.all(np.isnan(res["beta"][:4]))
    mask = np.ones((N, GAMMA), np.uint8)
    mask[10:14] = 0
    res = oracle.sts_fit(z, a, mask)
    assert np.all(res["status"] == 0)
    np.testing.assert_allclose(res["beta"], 1.0, rtol=1e-5)
