"""Pins of the oracle's gradient of the statistics' loss numerators
(0.1 CE + 0.9 L1 + 1.0 BCE, position-weighted and masked; the target and the
BCE label accept held fixed) against finite differences of the oracle's own
forward numerators, float64 autograd of the same objective written with
library routines, and closed forms."""
import numpy as np
import pytest
import torch


def _inputs(N, gamma, V, seed, rho=0.5):
    rng = np.random.default_rng(seed)
    t = rng.normal(0, 2, (N, gamma, V)).astype(np.float32)
    d = (rho * t + np.sqrt(1 - rho * rho) * rng.normal(0, 2, (N, gamma, V))).astype(np.float32)
    y = rng.integers(0, V, (N, gamma)).astype(np.int32)
    zc = rng.normal(0, 1, (N, gamma)).astype(np.float32)
    return d, t, y, zc


def test_backward_finite_differences(oracle):
    """Central differences of the forward numerators (V = 16): 0.1 CE + 0.9 L1
    in the draft logits, BCE in the confidence logit."""
    N, gamma, V = 2, 3, 16
    d, t, y, zc = _inputs(N, gamma, V, 11)
    mask = np.ones((N, gamma), np.uint8)
    mask[1, 2] = 0
    gd, gc = oracle.accept_stats_backward(d, t, y, zc, mask)
    h = 2.0 ** -14

    def j_draft(dd):
        ln = oracle.accept_stats(dd, t, y, zc, mask)["loss_num"]
        return 0.1 * ln[0] + 0.9 * ln[1]

    for (n, k, v) in [(0, 0, 3), (0, 1, 0), (0, 2, 15), (1, 0, 7), (1, 1, int(y[1, 1])), (1, 2, 5)]:
        dp, dm = d.copy(), d.copy()
        dp[n, k, v] = np.float32(d[n, k, v] + h)
        dm[n, k, v] = np.float32(d[n, k, v] - h)
        fd = (j_draft(dp) - j_draft(dm)) / (float(dp[n, k, v]) - float(dm[n, k, v]))
        assert abs(fd - gd[n, k, v]) < 1e-5 + 1e-3 * abs(fd), (n, k, v, fd, gd[n, k, v])
    for (n, k) in [(0, 0), (0, 2), (1, 1), (1, 2)]:
        zp, zm = zc.copy(), zc.copy()
        zp[n, k] = np.float32(zc[n, k] + h)
        zm[n, k] = np.float32(zc[n, k] - h)
        fd = (oracle.accept_stats(d, t, y, zp, mask)["loss_num"][2] -
              oracle.accept_stats(d, t, y, zm, mask)["loss_num"][2]) / (float(zp[n, k]) - float(zm[n, k]))
        assert abs(fd - gc[n, k]) < 1e-6 + 1e-4 * abs(fd), (n, k, fd, gc[n, k])
    assert np.all(gd[1, 2] == 0.0) and gc[1, 2] == 0.0  # masked position


def test_backward_matches_float64_autograd(oracle):
    """The same objective in float64 torch (softmax, log_softmax, softplus,
    abs; accept detached), differentiated by autograd; a scale of 0.25."""
    N, gamma, V = 3, 4, 64
    d, t, y, zc = _inputs(N, gamma, V, 12, rho=0.9)
    mask = (np.arange(N * gamma).reshape(N, gamma) % 5 != 3).astype(np.uint8)
    gd, gc = oracle.accept_stats_backward(d, t, y, zc, mask, scale=0.25)
    D = torch.tensor(d, dtype=torch.float64, requires_grad=True)
    Z = torch.tensor(zc, dtype=torch.float64, requires_grad=True)
    Tt = torch.tensor(t, dtype=torch.float64)
    pd, pt = torch.softmax(D, -1), torch.softmax(Tt, -1)
    ce = -torch.log_softmax(D, -1).gather(-1, torch.tensor(y, dtype=torch.int64)[..., None])[..., 0]
    l1 = (pd - pt).abs().sum(-1)
    acc = (1 - l1 / 2).clamp(0, 1).detach()
    bce = torch.nn.functional.softplus(Z) - acc * Z
    w = torch.exp(-torch.arange(1, gamma + 1, dtype=torch.float64) / gamma)
    m = torch.tensor(mask, dtype=torch.float64)
    J = 0.25 * (m * w * (0.1 * ce + 0.9 * l1 + 1.0 * bce)).sum()
    J.backward()
    np.testing.assert_allclose(gd, D.grad.numpy(), atol=1e-7, rtol=1e-5)
    np.testing.assert_allclose(gc, Z.grad.numpy(), atol=1e-7, rtol=1e-5)


def test_backward_closed_forms(oracle):
    """Identical rows: the L1 part vanishes (every sign is 0), so the draft
    gradient is 0.1 w (softmax - one-hot(label)); a one-hot draft row far from
    the target: L1 near 2, accept 0, BCE gradient w sigmoid(z)."""
    N, gamma, V = 1, 2, 32
    d, _, y, zc = _inputs(N, gamma, V, 13)
    gd, gc = oracle.accept_stats_backward(d, d.copy(), y, zc)
    for k in range(gamma):
        w = np.exp(-(k + 1) / gamma)
        p = torch.softmax(torch.tensor(d[0, k], dtype=torch.float64), 0).numpy()
        onehot = np.eye(V)[y[0, k]]
        np.testing.assert_allclose(gd[0, k], 0.1 * w * (p - onehot), atol=1e-8, rtol=1e-6)
        np.testing.assert_allclose(gc[0, k], w * (1 / (1 + np.exp(-float(zc[0, k]))) - 1.0), rtol=1e-6)
    dd = np.full((1, 1, V), -1e4, np.float32)
    tt = np.full((1, 1, V), -1e4, np.float32)
    dd[0, 0, 3], tt[0, 0, 9] = 0.0, 0.0
    _, gc2 = oracle.accept_stats_backward(dd, tt, np.array([[3]], np.int32), np.array([[0.7]], np.float32))
    assert abs(gc2[0, 0] - np.exp(-1.0) / (1 + np.exp(-0.7))) < 1e-7


def test_backward_bad_inputs(oracle):
    """A label outside [0, V) or a NaN logit: a NaN gradient row (and NaN
    confidence gradient); masked, the same positions give exact zeros."""
    N, gamma, V = 1, 3, 16
    d, t, y, zc = _inputs(N, gamma, V, 14)
    y[0, 1] = V
    d[0, 2, 5] = np.nan
    gd, gc = oracle.accept_stats_backward(d, t, y, zc)
    assert np.all(np.isfinite(gd[0, 0])) and np.all(np.isnan(gd[0, 1])) and np.all(np.isnan(gd[0, 2]))
    assert np.isnan(gc[0, 1]) and np.isnan(gc[0, 2])
    gd, gc = oracle.accept_stats_backward(d, t, y, zc, np.array([[1, 0, 0]], np.uint8))
    assert np.all(gd[0, 1:] == 0.0) and np.all(gc[0, 1:] == 0.0)
