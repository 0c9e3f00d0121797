"""GPU parity of the Sequential Temperature Scaling fit (dspark_sts_fit)
against the oracle.

Statuses are compared exactly; beta within 1e-5 relative.  The device sums
the pair terms in fp32 per thread and fp64 across threads, and stops its
Newton search once a step is below 1e-7 of beta, so it agrees with the
oracle's bisection to about 1e-7; 1e-5 leaves a margin of 100."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
RTOL = 1e-5


@pytest.fixture(scope="module")
def ds():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import verify_dspark_markov_gb300 as ds
    from verify_dspark_markov_gb300 import build
    build.build()
    ds.load()
    return ds


def _both(ds, oracle, z, a, mask=None):
    ref = oracle.sts_fit(z, a, mask)
    dev = torch.device("cuda")
    beta, status, passes = ds.sts_fit(torch.from_numpy(z).to(dev), torch.from_numpy(a).to(dev),
                                      None if mask is None else torch.from_numpy(mask).to(dev))
    torch.cuda.synchronize()
    # every position stops well inside the enqueued passes
    assert int(passes.max()) < 64
    return ref, beta.cpu().numpy(), status.cpu().numpy()


def _check(ref, beta, status):
    np.testing.assert_array_equal(status, ref["status"])
    fin = np.isfinite(ref["beta"])
    np.testing.assert_allclose(beta[fin], ref["beta"][fin], rtol=RTOL, atol=0)
    assert np.all(np.isnan(beta[~fin]))


def test_sts_soft_labels(ds, oracle):
    rng = np.random.default_rng(11)
    z = rng.normal(0, 2.0, (200_000, 5)).astype(np.float32)
    T = np.array([0.25, 0.5, 1.0, 2.0, 7.0])
    a = (1.0 / (1.0 + np.exp(-z.astype(np.float64) / T))).astype(np.float32)
    ref, beta, status = _both(ds, oracle, z, a)
    _check(ref, beta, status)
    np.testing.assert_allclose(beta, 1.0 / T, rtol=RTOL)


def test_sts_bernoulli_labels_with_mask(ds, oracle):
    """A million logged blocks of gamma = 7: hard accept labels drawn from a
    miscalibrated confidence, 30 % of the pairs masked."""
    rng = np.random.default_rng(12)
    N, G = 1_000_000, 7
    z = rng.normal(0, 2.0, (N, G)).astype(np.float32)
    true_T = np.linspace(0.6, 3.0, G)
    a = (rng.random((N, G)) < 1.0 / (1.0 + np.exp(-z / true_T))).astype(np.float32)
    mask = (rng.random((N, G)) < 0.7).astype(np.uint8)
    _check(*_both(ds, oracle, z, a, mask))


def test_sts_degenerate_and_invalid_positions(ds, oracle):
    """No information, separated labels, anti-correlated labels (beta 0), a
    fully masked position, a fitted one; then invalid pairs (status 3)."""
    rng = np.random.default_rng(13)
    N, G = 100_000, 6
    z = rng.normal(0, 2.0, (N, G)).astype(np.float32)
    a = rng.random((N, G)).astype(np.float32)
    z[:, 0] = 0.0
    a[:, 1] = (z[:, 1] > 0)
    a[:, 2] = (z[:, 2] < 0)
    a[:, 4] = 1.0 / (1.0 + np.exp(-z[:, 4]))
    a[:, 5] = np.where(z[:, 5] > 0, 1.0 / (1.0 + np.exp(-z[:, 5])), 0.0)  # nearly separated: finite
    mask = np.ones((N, G), np.uint8)
    mask[:, 3] = 0
    ref, beta, status = _both(ds, oracle, z, a.astype(np.float32), mask)
    assert ref["status"].tolist() == [1, 2, 0, 1, 0, 0]
    _check(ref, beta, status)
    z[5, 0] = np.nan
    a[6, 4] = 1.25
    ref, beta, status = _both(ds, oracle, z, a.astype(np.float32), mask)
    assert ref["status"].tolist() == [3, 2, 0, 1, 3, 0]
    _check(ref, beta, status)


def test_sts_large_beta_and_empty(ds, oracle):
    """A sharp confidence (beta near 1e4) and an empty log (N = 0)."""
    rng = np.random.default_rng(14)
    z = rng.normal(0, 0.01, (200_000, 2)).astype(np.float32)
    a = (1.0 / (1.0 + np.exp(-np.clip(z.astype(np.float64) / np.array([1e-4, 3e-3]), -700, 700)))).astype(np.float32)
    _check(*_both(ds, oracle, z, a))
    ref, beta, status = _both(ds, oracle, np.zeros((0, 4), np.float32), np.zeros((0, 4), np.float32))
    assert status.tolist() == [1, 1, 1, 1] and beta.tolist() == [1.0] * 4
    _check(ref, beta, status)


def test_sts_repeat_is_bitwise_identical(ds):
    """The CTAs' sums are combined in a fixed order: two fits of the same
    log give the same bits."""
    rng = np.random.default_rng(15)
    z = torch.from_numpy(rng.normal(0, 2.0, (3_000_000, 7)).astype(np.float32)).cuda()
    a = (torch.rand(z.shape, device="cuda") < torch.sigmoid(z / 1.7)).float()
    b1, s1, p1 = ds.sts_fit(z, a)
    b2, s2, p2 = ds.sts_fit(z, a)
    torch.cuda.synchronize()
    assert torch.equal(b1.view(torch.int64), b2.view(torch.int64))
    assert torch.equal(s1, s2) and torch.equal(p1, p2)
    assert torch.all(s1 == 0)


def test_sts_pass_budget_exhausted(ds, oracle):
    """Two passes leave every informative position searching (the first pass
    is taken at beta = 0, the second starts Newton at beta = 1): they report
    status 4 with their last iterate, which the default budget carries on to
    the oracle's fit."""
    rng = np.random.default_rng(16)
    z = rng.normal(0, 2.0, (200_000, 5)).astype(np.float32)
    T = np.array([0.25, 0.5, 3.0, 2.0, 7.0])
    a = (1.0 / (1.0 + np.exp(-z.astype(np.float64) / T))).astype(np.float32)
    zd, ad = torch.from_numpy(z).cuda(), torch.from_numpy(a).cuda()
    beta, status, passes = ds.sts_fit(zd, ad, max_passes=2)
    torch.cuda.synchronize()
    assert status.tolist() == [4] * 5 and passes.tolist() == [2] * 5
    assert np.all(np.isfinite(beta.cpu().numpy()))
    ref = oracle.sts_fit(z, a)
    beta, status, passes = ds.sts_fit(zd, ad)
    torch.cuda.synchronize()
    _check(ref, beta.cpu().numpy(), status.cpu().numpy())


def test_sts_ragged_rows_and_misaligned_inputs(ds, oracle):
    """Row counts that leave one to three rows after the four-row chunks the
    kernel reads as vectors, and inputs that start off a 16-byte boundary
    (read a row at a time): the same fit as the oracle's."""
    rng = np.random.default_rng(17)
    for N, G in ((10_007, 7), (50_001, 3), (3, 5)):
        z = rng.normal(0, 2.0, (N, G)).astype(np.float32)
        a = (rng.random((N, G)) < 1.0 / (1.0 + np.exp(-z / 1.3))).astype(np.float32)
        mask = (rng.random((N, G)) < 0.8).astype(np.uint8)
        if N == 3:  # three rows cannot pin a fit down: soft labels keep it finite
            a = (1.0 / (1.0 + np.exp(-z / 1.3))).astype(np.float32)
            mask[:] = 1
        _check(*_both(ds, oracle, z, a, mask))
    # views one element into larger buffers: 4-byte aligned, not 16
    N, G = 40_000, 4
    z = rng.normal(0, 2.0, (N, G)).astype(np.float32)
    a = (1.0 / (1.0 + np.exp(-z.astype(np.float64) / np.array([0.5, 1.0, 2.0, 4.0])))).astype(np.float32)
    mask = (rng.random((N, G)) < 0.9).astype(np.uint8)
    ref = oracle.sts_fit(z, a, mask)
    dev = torch.device("cuda")
    zb = torch.zeros(N * G + 1, dtype=torch.float32, device=dev)
    ab = torch.zeros(N * G + 1, dtype=torch.float32, device=dev)
    mb = torch.zeros(N * G + 1, dtype=torch.uint8, device=dev)
    zb[1:] = torch.from_numpy(z.reshape(-1)).to(dev)
    ab[1:] = torch.from_numpy(a.reshape(-1)).to(dev)
    mb[1:] = torch.from_numpy(mask.reshape(-1)).to(dev)
    zv, av, mv = zb[1:].view(N, G), ab[1:].view(N, G), mb[1:].view(N, G)
    assert zv.data_ptr() % 16 != 0 and mv.data_ptr() % 4 != 0
    beta, status, passes = ds.sts_fit(zv, av, mv)
    torch.cuda.synchronize()
    _check(ref, beta.cpu().numpy(), status.cpu().numpy())
    np.testing.assert_allclose(beta.cpu().numpy(), [2.0, 1.0, 0.5, 0.25], rtol=1e-3)
